// The streaming tcgen05 expand kernel for 128-token tiles (see lora_stream.cuh).
#include "lora_stream.cuh"

namespace csgmv {

struct StBars {
    uint64_t *b_full, *b_empty, *y_full, *y_empty;  // [S]
    uint64_t *acc_full, *acc_empty;                 // [kStAcc]
    uint64_t *op_full, *op_empty;                   // [2]
    uint32_t *tmem_slot;
    int *tok;   // [2][128] token of each tile row (-1: none)
    int *flag;  // [2] the tile's rows are consecutive tokens; [2, 4) scratch
};

__device__ __forceinline__ StBars st_bars(const StreamParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    StBars w;
    w.b_full = b;
    w.b_empty = b + k.S;
    w.y_full = b + 2 * k.S;
    w.y_empty = b + 3 * k.S;
    w.acc_full = b + 4 * k.S;
    w.acc_empty = w.acc_full + kStAcc;
    w.op_full = w.acc_empty + kStAcc;
    w.op_empty = w.op_full + 2;
    w.tmem_slot = reinterpret_cast<uint32_t *>(w.op_empty + 2);
    w.tok = reinterpret_cast<int *>(smem + k.o_tok);
    w.flag = w.tok + 256;
    return w;
}

struct StUnit {
    int w, p0, M;  // slot, first sorted position, tokens of the tile
    int j, n0, n1, nt;  // slice, columns [n0, n1), stages
};

// Unit u of the walk (identical on every role).  False when the unit has no
// tensor-core work: a rank-0 slot (r = 0) or an invalid slot / rank (r < 0).
__device__ __forceinline__ bool st_unit(const StreamParams &k, const int *tables, int nruns, int64_t u, bool report,
                                        StUnit &U, int &r) {
    const LoraParams &p = k.p;
    const int tile = (int)(u / k.upt);
    int rem = (int)(u % k.upt);
    const Unit T = tile_of<128>(tables, k.runcap, nruns, tile);
    U.w = T.w;
    U.p0 = T.p0;
    U.M = T.M;
    int j = 0;
    for (; j + 1 < p.c; ++j) {
        const int nb = (p.off[j + 1] - p.off[j] + k.cb - 1) / k.cb;
        if (rem < nb) break;
        rem -= nb;
    }
    U.j = j;
    U.n0 = p.off[j] + rem * k.cb;
    U.n1 = min(p.off[j + 1], U.n0 + k.cb);
    U.nt = U.n1 > U.n0 ? (U.n1 - U.n0 + kStCols - 1) / kStCols : 0;
    r = unit_rank(p, T, report);
    return r > 0 && U.nt > 0;
}

// ------------------------------------------------------------------------------------- producer
__device__ void st_producer(const StreamParams &k, unsigned char *smem, const int *tables, int nruns,
                            int64_t nunits) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const StBars W = st_bars(k, smem);
    const uint32_t Bbytes = (uint32_t)kStCols * p.R * 2;
    uint32_t g = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, false, U, r)) continue;
        const int b = uc & 1;
        mbar_wait(&W.op_full[b], (uc >> 1) & 1, p.status, kStatusTimeout);
        const int *tok = W.tok + b * 128;
        const bool contig = W.flag[b] != 0;
        const int t0 = tok[0];
        const int tfill = t0 >= 0 ? t0 : 0;
        // row in the 2-D view of B_j of column x of the unit's slice
        const int brow = U.w * p.b_rows[U.j] + p.b_row0[U.j] - p.off[U.j];
        for (int i = 0; i < U.nt; ++i, ++g) {
            const int s = g % k.S;
            const uint32_t ph = (g / k.S) & 1;
            mbar_wait(&W.y_empty[s], ph ^ 1, p.status, kStatusTimeout);
            mbar_wait(&W.b_empty[s], ph ^ 1, p.status, kStatusTimeout);
            unsigned char *slot = smem + k.o_ring + s * k.slot_bytes;
            const int x0 = U.n0 + i * kStCols;
            if (lane == 0) {
                mbar_arrive_expect_tx(&W.b_full[s], Bbytes);
                tma_load_2d(slot + kStTileBytes, &k.tmB[U.j], 0, brow + x0, &W.b_full[s]);
                mbar_arrive_expect_tx(&W.y_full[s], p.accumulate ? kStTileBytes : 0);
                if (p.accumulate && contig) tma_load_2d(slot, &k.tmY, x0, t0, &W.y_full[s]);
            }
            if (p.accumulate && !contig) {
                // lane l: tile rows 4l .. 4l+3 in one gather; rows past the tile
                // (or of an invalid token) read a valid row that is never used
                __syncwarp();  // after the byte count is posted
                const int m = 4 * lane;
                auto grow = [&](int mm) {
                    const int t = mm < U.M ? tok[mm] : -1;
                    return t >= 0 ? t : tfill;
                };
                tma_gather4(slot + m * 128, &k.tmYg, x0, grow(m), grow(m + 1), grow(m + 2), grow(m + 3),
                            &W.y_full[s]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.op_empty[b]);  // done with the token list
        ++uc;
    }
}

// ------------------------------------------------------------------------------------- MMA issuer
__device__ void st_mma(const StreamParams &k, unsigned char *smem, const int *tables, int nruns, int64_t nunits,
                       uint32_t tmem) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const StBars W = st_bars(k, smem);
    const int Rb = p.R * 2;
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    const uint32_t op0 = smem_u32(smem + k.o_op);
    uint32_t g = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, false, U, r)) continue;
        const int b = uc & 1;
        mbar_wait(&W.op_full[b], (uc >> 1) & 1, p.status, kStatusTimeout);
        tc_fence_after();
        const int RK = (r + 15) & ~15;
        const int ksteps = RK / 16;
        const uint32_t ahi = op0 + (uint32_t)(2 * b) * kStTileBytes, alo = ahi + kStTileBytes;
        for (int i = 0; i < U.nt; ++i, ++g) {
            const int s = g % k.S;
            const int a = g % kStAcc;
            mbar_wait(&W.b_full[s], (g / k.S) & 1, p.status, kStatusTimeout);
            unsigned char *bs = smem + k.o_ring + s * k.slot_bytes + kStTileBytes;
            if (RK != r) {  // B columns [r, RK) are adapter padding (even NaN): zero them
                const int c0 = r >> 3, nc = (RK >> 3) - c0;
                for (int idx = lane; idx < kStCols * nc; idx += 32) {
                    const int n = idx / nc, ch = c0 + idx % nc;
                    uint16_t *q16 = reinterpret_cast<uint16_t *>(bs) + swz(n, ch, pcB, shB);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (ch * 8 + e >= r) q16[e] = 0;
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            mbar_wait(&W.acc_empty[a], ((g / kStAcc) & 1) ^ 1, p.status, kStatusTimeout);
            tc_fence_after();
            if (lane == 0) {
                const int x0 = U.n0 + i * kStCols;
                const int ncols = min(U.n1, x0 + kStCols) - x0;
                const uint32_t idesc = idesc_bf16_f32(128, (ncols + 15) & ~15);
                const uint32_t bsa = smem_u32(bs);
                const uint32_t d = tmem + (uint32_t)(a * kStCols);
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint64_t bd = smem_desc_kmajor(bsa + ks * 32, Rb);
                    tc_mma_bf16(d, smem_desc_kmajor(ahi + ks * 32, 128), bd, idesc, ks > 0);
                    tc_mma_bf16(d, smem_desc_kmajor(alo + ks * 32, 128), bd, idesc, true);
                }
                tc_commit(&W.b_empty[s]);
                tc_commit(&W.acc_full[a]);
            }
            __syncwarp();
        }
        ++uc;
    }
    // the last slot releases land before the CTA (and its barriers) goes away
    for (uint32_t gg = g > (uint32_t)k.S ? g - k.S : 0; gg < g; ++gg)
        mbar_wait(&W.b_empty[gg % k.S], (gg / k.S) & 1, p.status, kStatusTimeout);
}

// ------------------------------------------------------------------------------------- operands
// h[t][col .. col+7] as fp32 (0 past `r` columns of the slice, i.e. col >= lim).
__device__ __forceinline__ void st_h8(const LoraParams &p, int t, int col, int lim, float (&v)[8]) {
    const int64_t o = (int64_t)t * p.ldh + col;
    if (p.h_f32) {
        const float *h = reinterpret_cast<const float *>(p.h) + o;
        if (col + 8 <= lim && (o & 3) == 0) {
            const float4 a = *reinterpret_cast<const float4 *>(h), b = *reinterpret_cast<const float4 *>(h + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = col + e < lim ? h[e] : 0.f;
        }
    } else {
        const __nv_bfloat16 *h = reinterpret_cast<const __nv_bfloat16 *>(p.h) + o;
        if (col + 8 <= lim && (o & 7) == 0) {
            const uint4 a = *reinterpret_cast<const uint4 *>(h);
            float2 f;
            f = unpack_bf16x2(a.x); v[0] = f.x; v[1] = f.y;
            f = unpack_bf16x2(a.y); v[2] = f.x; v[3] = f.y;
            f = unpack_bf16x2(a.z); v[4] = f.x; v[5] = f.y;
            f = unpack_bf16x2(a.w); v[6] = f.x; v[7] = f.y;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = col + e < lim ? __bfloat162float(h[e]) : 0.f;
        }
    }
}

__device__ void st_operands(const StreamParams &k, unsigned char *smem, const int *tables, int nruns,
                            int64_t nunits) {
    const LoraParams &p = k.p;
    const int otid = threadIdx.x - 64, lane = otid & 31, ow = otid >> 5;
    const StBars W = st_bars(k, smem);
    uint32_t uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, otid == 0, U, r)) continue;
        const int b = uc & 1;
        mbar_wait(&W.op_empty[b], ((uc >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        int *tok = W.tok + b * 128;
        int tm[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int m = otid + 64 * h2;
            int t = -1;
            if (m < U.M) {
                t = p.permutation[U.p0 + m];
                if (t < 0 || t >= p.num_tokens) {
                    atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
                    t = -1;
                }
            }
            tok[m] = t;
            tm[h2] = t;
        }
        named_bar_sync(kStOpBar, 64);
        const int t0 = tok[0];
        bool mine = true;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int m = otid + 64 * h2;
            if (m < U.M) mine = mine && tm[h2] == t0 + m;
        }
        const bool wall = __all_sync(0xffffffffu, mine);
        if (lane == 0) W.flag[2 + ow] = wall ? 1 : 0;
        named_bar_sync(kStOpBar, 64);
        if (otid == 0) W.flag[b] = (W.flag[2] && W.flag[3] && t0 >= 0) ? 1 : 0;

        // operand tiles: row m = token m of the tile, columns [0, RK) of slice j
        unsigned char *ahi = smem + k.o_op + (2 * b) * kStTileBytes;
        unsigned char *alo = ahi + kStTileBytes;
        const int RK = (r + 15) & ~15;
        const int col0 = U.j * r;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int m = otid + 64 * h2;
            const int t = tm[h2];
            for (int ch = 0; ch < RK / 8; ++ch) {
                float v[8];
                if (t >= 0) {
                    st_h8(p, t, col0 + ch * 8, col0 + r, v);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.f;
                }
                uint4 hi, lo;
                split_pair(v[0], v[1], hi.x, lo.x);
                split_pair(v[2], v[3], hi.y, lo.y);
                split_pair(v[4], v[5], hi.z, lo.z);
                split_pair(v[6], v[7], hi.w, lo.w);
                const int off = m * 128 + ((ch ^ (m & 7)) << 4);
                *reinterpret_cast<uint4 *>(ahi + off) = hi;
                *reinterpret_cast<uint4 *>(alo + off) = lo;
            }
        }
        fence_proxy_async_smem();  // the operand tiles are read by the tensor core
        named_bar_sync(kStOpBar, 64);
        if (otid == 0) mbar_arrive(&W.op_full[b]);
        ++uc;
    }
}

// ------------------------------------------------------------------------------------- epilogue
__device__ void st_epilogue(const StreamParams &k, unsigned char *smem, const int *tables, int nruns,
                            int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int team = (warp - kStEpiWarp0) >> 2;
    const int q = warp & 3;  // TMEM lanes (tile rows) 32q .. 32q+31
    const int row = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const StBars W = st_bars(k, smem);
    uint32_t g = 0, uc = 0;
    int pending = -1;  // lane 0: the slot of this warp's last box store, not yet handed back
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, false, U, r)) {
            // a non-accumulating expand of a rank-0 slot writes a zero delta
            if (r == 0 && !p.accumulate && team == 0 && row < U.M) {
                const int t = p.permutation[U.p0 + row];
                if (t >= 0 && t < p.num_tokens)
                    for (int col = U.n0; col < U.n1; col += 8)
                        *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
        const int b = uc & 1;
        mbar_wait(&W.op_full[b], (uc >> 1) & 1, p.status, kStatusTimeout);
        const int *tok = W.tok + b * 128;
        const bool box = W.flag[b] != 0 && U.M == 128;
        const int t0 = tok[0];
        const int trow = row < U.M ? tok[row] : -1;
        const float sigma = p.scalings[U.w];
        for (int i = 0; i < U.nt; ++i, ++g) {
            if ((int)(g & 1) != team) continue;
            const int s = g % k.S;
            const int a = g % kStAcc;
            mbar_wait(&W.acc_full[a], (g / kStAcc) & 1, p.status, kStatusTimeout);
            mbar_wait(&W.y_full[s], (g / k.S) & 1, p.status, kStatusTimeout);
            tc_fence_after();
            __syncwarp();  // tcgen05.ld is warp-wide
            float v[2][32];
            tmem_ld32(tmem + lane_base + (uint32_t)(a * kStCols), v[0]);
            tmem_ld32(tmem + lane_base + (uint32_t)(a * kStCols + 32), v[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&W.acc_empty[a]);
            const int x0 = U.n0 + i * kStCols;
            const int ncols = min(U.n1, x0 + kStCols) - x0;
            const bool full = box && ncols == kStCols;
            unsigned char *ys = smem + k.o_ring + s * k.slot_bytes;
            if (row < U.M && (full || trow >= 0)) {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    if (8 * c8 < ncols) {
                        uint4 *ptr = reinterpret_cast<uint4 *>(ys + row * 128 + ((c8 ^ (row & 7)) << 4));
                        const float *vv = &v[c8 >> 2][8 * (c8 & 3)];
                        uint4 bv = p.accumulate ? *ptr : make_uint4(0, 0, 0, 0);
                        float2 f;
                        f = unpack_bf16x2(bv.x); bv.x = pack_bf16x2(f.x + sigma * vv[0], f.y + sigma * vv[1]);
                        f = unpack_bf16x2(bv.y); bv.y = pack_bf16x2(f.x + sigma * vv[2], f.y + sigma * vv[3]);
                        f = unpack_bf16x2(bv.z); bv.z = pack_bf16x2(f.x + sigma * vv[4], f.y + sigma * vv[5]);
                        f = unpack_bf16x2(bv.w); bv.w = pack_bf16x2(f.x + sigma * vv[6], f.y + sigma * vv[7]);
                        if (full) *ptr = bv;
                        else *reinterpret_cast<uint4 *>(p.y + (int64_t)trow * p.N + x0 + 8 * c8) = bv;
                    }
                }
            }
            if (full) {
                fence_proxy_async_smem();  // the in-place rows before the TMA store reads them
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&k.tmYs, x0, t0 + 32 * q, ys + 32 * q * 128);
                    bulk_commit();
                    if (pending >= 0) {  // the previous store has read its rows: hand its slot back
                        bulk_wait_read<1>();
                        mbar_arrive(&W.y_empty[pending]);
                    }
                    pending = s;
                }
            } else {
                fence_proxy_async_smem();  // this warp's reads of the slot before a TMA refills it
                __syncwarp();
                if (lane == 0) {
                    if (pending >= 0) {
                        bulk_wait_read<0>();
                        mbar_arrive(&W.y_empty[pending]);
                        pending = -1;
                    }
                    mbar_arrive(&W.y_empty[s]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.op_empty[b]);  // done with the token list (and its MMAs, see below)
        ++uc;
    }
    if (lane == 0) bulk_wait<0>();  // every store has completed before the CTA ends
}

// The operand tiles of a unit are free once every epilogue warp has finished
// the unit: the team that took the unit's last stage waited for that stage's
// accumulator, i.e. for every MMA of the unit.
__global__ void __launch_bounds__(kStThreads, 1) lora_stream_expand_kernel(const __grid_constant__ StreamParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const StBars W = st_bars(k, smem);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < k.S; ++i) {
            mbar_init(&W.b_full[i], 1);
            mbar_init(&W.b_empty[i], 1);
            mbar_init(&W.y_full[i], 1);
            mbar_init(&W.y_empty[i], 4);  // the four warps of the team that takes the stage
        }
        for (int i = 0; i < kStAcc; ++i) {
            mbar_init(&W.acc_full[i], 1);
            mbar_init(&W.acc_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&W.op_full[i], 1);
            mbar_init(&W.op_empty[i], 1 + 8);  // producer + epilogue warps
        }
        fence_mbar_init();
        for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmB[j]);
        prefetch_tmap(&k.tmY);
        prefetch_tmap(&k.tmYs);
        prefetch_tmap(&k.tmYg);
    }
    if (warp == 1) {  // one warp owns the TMEM accumulators of the CTA
        tmem_alloc(W.tmem_slot, kStAcc * kStCols);
        tmem_relinquish();
    }
    tc_fence_before();
    int nruns = 0;
    int *tables = reinterpret_cast<int *>(smem + k.o_run);
    const int ntiles = build_run_table_raw<128>(k.p, k.max_segments, k.runcap, tables, &nruns);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = *W.tmem_slot;
    const int64_t nunits = (int64_t)ntiles * k.upt;
    if (warp == 0) st_producer(k, smem, tables, nruns, nunits);
    else if (warp == 1) st_mma(k, smem, tables, nruns, nunits, tmem);
    else if (warp < kStEpiWarp0) st_operands(k, smem, tables, nruns, nunits);
    else st_epilogue(k, smem, tables, nruns, nunits, tmem);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kStAcc * kStCols);
    }
}

const void *lora_kernel_stream() { return reinterpret_cast<const void *>(lora_stream_expand_kernel); }

}  // namespace csgmv
