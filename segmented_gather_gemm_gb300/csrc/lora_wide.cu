// The wide-output expand for short slot runs (see lora_wide.cuh).
#include "lora_wide.cuh"

namespace csgmv {
namespace {

struct WideBars {
    uint64_t *full, *done, *empty;  // [S] each (done: unused)
};

__device__ __forceinline__ WideBars wide_bars(const WideParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    return WideBars{b, b + k.S, b + 2 * k.S};
}

// One unit: tile `u / nblk`, column block `u % nblk`, columns [x0, x1), in
// nst stages.  False when nothing is written (an invalid slot or rank, or
// rank 0 with accumulate).  Identical on every thread.
struct WUnit {
    int w, p0, M, r, x0, x1, nst;
};

template <int TM>
__device__ __forceinline__ bool wide_unit(const WideParams &k, const int *tables, int nruns, int nblk, int u,
                                          bool report, WUnit &U) {
    const LoraParams &p = k.p;
    const Unit T = tile_of<TM>(tables, k.runcap, nruns, u / nblk);
    const int blk = u - (u / nblk) * nblk;
    U.w = T.w;
    U.p0 = T.p0;
    U.M = T.M;
    U.r = unit_rank(p, T, report && blk == 0);
    U.x0 = p.off[0] + blk * k.cb;
    U.x1 = min(p.off[p.c], U.x0 + k.cb);
    U.nst = (U.x1 - U.x0 + k.nt - 1) / k.nt;
    return U.M > 0 && U.x1 > U.x0 && (U.r > 0 || (U.r == 0 && !p.accumulate));
}

// Token of row `row` of the unit's tile, or -1 (past the tile or out of range).
__device__ __forceinline__ int wide_token(const LoraParams &p, const WUnit &U, int row) {
    if (row >= U.M) return -1;
    const int t = p.permutation[U.p0 + row];
    return t >= 0 && t < p.num_tokens ? t : -1;
}

// ------------------------------------------------------------------------------------------ load
template <int TM>
__device__ void wide_load(const WideParams &k, unsigned char *smem, const int *tables, int nruns, int nblk,
                          int units) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const WideBars W = wide_bars(k, smem);
    const int R = p.R;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        WUnit U;
        if (!wide_unit<TM>(k, tables, nruns, nblk, u, lane == 0, U)) continue;
        const int t = lane < TM ? wide_token(p, U, lane) : -1;
        if (lane < U.M && t < 0) atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
        const bool row_copy = t >= 0 && p.accumulate;
        const int nrows = __popc(__ballot_sync(0xffffffffu, row_copy));
        for (int st = 0; st < U.nst; ++st, ++it) {
            const int s = it % k.S;
            mbar_wait(&W.empty[s], ((it / k.S) & 1) ^ 1, p.status, kStatusTimeout);
            unsigned char *stg = smem + k.o_ring + s * k.stage_bytes;
            const int c0 = U.x0 + st * k.nt, c1 = min(U.x1, c0 + k.nt);
            if (lane == 0)
                mbar_arrive_expect_tx(&W.full[s], (uint32_t)k.nt * R * 2 + (uint32_t)nrows * (c1 - c0) * 2);
            __syncwarp();  // the byte count is posted before any copy can land
            if (lane == 0) {
                unsigned char *bs = stg + k.b_off;
                if (!p.b_tuple) {
                    for (int bb = 0; bb < k.nt; bb += 256)
                        tma_load_2d(bs + bb * R * 2, &k.tmB, 0, U.w * (int)p.N + c0 + bb, &W.full[s]);
                } else {
                    for (int bb = 0; bb < k.nt; bb += 64) {
                        const int col = c0 + bb;
                        const int j = (p.c > 1 && col >= p.off[1]) + (p.c > 2 && col >= p.off[2]);
                        tma_load_2d(bs + bb * R * 2, &k.tmBs[j], 0, U.w * p.b_rows[j] + p.b_row0[j] + (col - p.off[j]),
                                    &W.full[s]);
                    }
                }
            }
            if (row_copy) bulk_g2s(stg + lane * k.ypitch, p.y + (int64_t)t * p.N + c0, (uint32_t)(c1 - c0) * 2, &W.full[s]);
        }
    }
}

// --------------------------------------------------------------------------------------- consume
// h[t][col] summed over the workspace planes (one plane: h itself).
__device__ __forceinline__ float wide_h(const LoraParams &p, int t, int col) {
    float v = 0.f;
    const int parts = max(1, p.h_parts);
    for (int q = 0; q < parts; ++q) {
        const int64_t o = (int64_t)q * p.h_plane + (int64_t)t * p.ldh + col;
        v += p.h_f32 ? reinterpret_cast<const float *>(p.h)[o]
                     : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[o]);
    }
    return v;
}

template <int TM, int RMAX>
__device__ void wide_consume(const WideParams &k, unsigned char *smem, const int *tables, int nruns, int nblk,
                             int units, int cw) {
    constexpr int KS = RMAX / 16, NMT = TM / 16;
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const WideBars W = wide_bars(k, smem);
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    const int wcols = k.nt / kWideConsumers;  // this warp's columns of a stage: [lc0, lc0 + wcols)
    const int lc0 = cw * wcols;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        WUnit U;
        if (!wide_unit<TM>(k, tables, nruns, nblk, u, false, U)) continue;
        const float sigma = U.r > 0 ? p.scalings[U.w] : 0.f;
        const int ksteps = (U.r + 15) / 16;
        const bool r_ragged = U.r > 0 && (p.R == 8 ? (U.r < 8) : (U.r % 16 != 0));
        // tokens of the rows this lane's fragments hold: mt * 16 + lane / 4 (+ 8)
        int trow[NMT][2];
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) trow[mt][hh] = wide_token(p, U, mt * 16 + (lane >> 2) + 8 * hh);
        // h of one slice as bf16 hi / lo A fragments, every 16-row tile
        uint32_t fhi[NMT][KS][4], flo[NMT][KS][4];
        int cur = -1;
        auto load_slice = [&](int j) {
            // every value is loaded before any is split, so the loads overlap
            float v[NMT][KS][8];
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int kk = ks * 16 + 2 * (lane & 3) + (e & 1) + ((e & 4) ? 8 : 0);
                        const int t = trow[mt][(e >> 1) & 1];
                        v[mt][ks][e] = kk < U.r && t >= 0 ? wide_h(p, t, j * U.r + kk) : 0.f;
                    }
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    split_pair(v[mt][ks][0], v[mt][ks][1], fhi[mt][ks][0], flo[mt][ks][0]);
                    split_pair(v[mt][ks][2], v[mt][ks][3], fhi[mt][ks][1], flo[mt][ks][1]);
                    split_pair(v[mt][ks][4], v[mt][ks][5], fhi[mt][ks][2], flo[mt][ks][2]);
                    split_pair(v[mt][ks][6], v[mt][ks][7], fhi[mt][ks][3], flo[mt][ks][3]);
                }
            cur = j;
        };
        auto slice_of_col = [&](int col) { return (p.c > 1 && col >= p.off[1]) + (p.c > 2 && col >= p.off[2]); };
        for (int st = 0; st < U.nst; ++st, ++it) {
            const int s = it % k.S;
            mbar_wait(&W.full[s], (it / k.S) & 1, p.status, kStatusTimeout);
            unsigned char *ys = smem + k.o_ring + s * k.stage_bytes;
            __nv_bfloat16 *bs = reinterpret_cast<__nv_bfloat16 *>(ys + k.b_off);
            const uint32_t bs_u = smem_u32(bs);
            const int c0 = U.x0 + st * k.nt, c1 = min(U.x1, c0 + k.nt);
            if (r_ragged) {
                // B columns [r, 16 * ceil(r / 16)) (R = 8: [r, 8)) of this warp's
                // rows are adapter padding: zero them, so that even NaN there
                // never reaches the output
                const int rpad = p.R == 8 ? 8 : (U.r + 15) / 16 * 16;
                const int npad = rpad - U.r;
                for (int idx = lane; idx < wcols * npad; idx += 32) {
                    const int n = lc0 + idx / npad, kk = U.r + idx % npad;
                    bs[swz(n, kk >> 3, pcB, shB) + (kk & 7)] = __float2bfloat16_rn(0.f);
                }
                __syncwarp();
            }
            // this warp's columns of the stage, [lcs, lce)
            const int lcs = c0 + lc0, lce = min(c1, c0 + lc0 + wcols);
            if (lcs < lce && slice_of_col(lcs) == slice_of_col(lce - 1)) {
                // one slice (always so for one output projection): every pair's
                // MMAs first, then every pair's epilogue, so that the pairs'
                // dependency chains overlap
                const int npv = (lce - lcs + 15) >> 4;      // pairs holding columns (<= wcols / 16 <= 2)
                const bool last_full = ((lce - lcs) & 15) == 0;  // the last pair's second half holds columns
                float acc[2][NMT][2][4];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc[q][mt][h][e] = 0.f;
                if (U.r > 0) {
                    const int j = slice_of_col(lcs);
                    if (j != cur) load_slice(j);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        if (ks < ksteps) {
                            uint32_t bf[2][4];
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                if (q < npv) {
                                    const int lc = lc0 + 16 * q;
                                    if (RMAX == 16 && p.R == 8) {
                                        ldmatrix_x2(bf[q][0], bf[q][2], bs + (lc + 8 * ((lane >> 3) & 1) + (lane & 7)) * 8);
                                        bf[q][1] = 0u;
                                        bf[q][3] = 0u;
                                    } else {
                                        const int nrow = lc + 8 * (lane >> 4) + (lane & 7);
                                        ldmatrix_x4(bf[q][0], bf[q][1], bf[q][2], bf[q][3],
                                                    bs + swz(nrow, 2 * ks + ((lane >> 3) & 1), pcB, shB));
                                    }
                                }
                            }
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                if (q < npv) {
                                    const bool h1 = q < npv - 1 || last_full;
#pragma unroll
                                    for (int mt = 0; mt < NMT; ++mt) {
                                        mma_bf16_16816(acc[q][mt][0], fhi[mt][ks], bf[q][0], bf[q][1]);
                                        mma_bf16_16816(acc[q][mt][0], flo[mt][ks], bf[q][0], bf[q][1]);
                                        if (h1) {
                                            mma_bf16_16816(acc[q][mt][1], fhi[mt][ks], bf[q][2], bf[q][3]);
                                            mma_bf16_16816(acc[q][mt][1], flo[mt][ks], bf[q][2], bf[q][3]);
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
                // y = base + sigma * acc, stored from registers (a quad of lanes
                // writes 16 consecutive bytes of a row)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q >= npv) continue;
                    const bool h1 = q < npv - 1 || last_full;
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (h == 1 && !h1) continue;
#pragma unroll
                            for (int rr = 0; rr < 2; ++rr) {
                                const int t = trow[mt][rr];
                                if (t < 0) continue;
                                const int row = mt * 16 + (lane >> 2) + 8 * rr;
                                const int col = lc0 + 16 * q + 8 * h + 2 * (lane & 3);
                                const float2 bv = p.accumulate
                                                      ? unpack_bf16x2(*reinterpret_cast<const uint32_t *>(ys + row * k.ypitch + col * 2))
                                                      : make_float2(0.f, 0.f);
                                *reinterpret_cast<uint32_t *>(p.y + (int64_t)t * p.N + c0 + col) = pack_bf16x2(
                                    bv.x + sigma * acc[q][mt][h][2 * rr], bv.y + sigma * acc[q][mt][h][2 * rr + 1]);
                            }
                        }
                }
            } else
            for (int pc = 0; pc < wcols; pc += 16) {
                const int lc = lc0 + pc;  // local column of the pair
                if (c0 + lc >= c1) break;
                const bool has1 = c0 + lc + 8 < c1;
                float acc[NMT][2][4];
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[mt][h][e] = 0.f;
                if (U.r > 0) {
                    const int j0 = (p.c > 1 && c0 + lc >= p.off[1]) + (p.c > 2 && c0 + lc >= p.off[2]);
                    const int j1 = has1 ? (p.c > 1 && c0 + lc + 8 >= p.off[1]) + (p.c > 2 && c0 + lc + 8 >= p.off[2]) : j0;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // both halves in one pass when they share a slice
                        if (half == 1 && (j1 == j0 || !has1)) break;
                        const int jh = half == 0 ? j0 : j1;
                        if (jh != cur) load_slice(jh);
                        const bool do0 = half == 0, do1 = has1 && (half == 1 || j1 == j0);
#pragma unroll
                        for (int ks = 0; ks < KS; ++ks) {
                            if (ks < ksteps) {
                                uint32_t bf[4];
                                if (RMAX == 16 && p.R == 8) {
                                    ldmatrix_x2(bf[0], bf[2], bs + (lc + 8 * ((lane >> 3) & 1) + (lane & 7)) * 8);
                                    bf[1] = 0u;
                                    bf[3] = 0u;
                                } else {
                                    const int nrow = lc + 8 * (lane >> 4) + (lane & 7);
                                    ldmatrix_x4(bf[0], bf[1], bf[2], bf[3],
                                                bs + swz(nrow, 2 * ks + ((lane >> 3) & 1), pcB, shB));
                                }
#pragma unroll
                                for (int mt = 0; mt < NMT; ++mt) {
                                    if (do0) {
                                        mma_bf16_16816(acc[mt][0], fhi[mt][ks], bf[0], bf[1]);
                                        mma_bf16_16816(acc[mt][0], flo[mt][ks], bf[0], bf[1]);
                                    }
                                    if (do1) {
                                        mma_bf16_16816(acc[mt][1], fhi[mt][ks], bf[2], bf[3]);
                                        mma_bf16_16816(acc[mt][1], flo[mt][ks], bf[2], bf[3]);
                                    }
                                }
                            }
                        }
                    }
                }
                // y = base + sigma * acc, stored from registers: a quad of lanes
                // writes 16 consecutive bytes of a row
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1 && !has1) continue;
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int row = mt * 16 + (lane >> 2) + 8 * rr;
                            const int t = trow[mt][rr];
                            if (t < 0) continue;
                            const int col = lc + 8 * h + 2 * (lane & 3);
                            const float2 bv = p.accumulate
                                                  ? unpack_bf16x2(*reinterpret_cast<const uint32_t *>(ys + row * k.ypitch + col * 2))
                                                  : make_float2(0.f, 0.f);
                            *reinterpret_cast<uint32_t *>(p.y + (int64_t)t * p.N + c0 + col) =
                                pack_bf16x2(bv.x + sigma * acc[mt][h][2 * rr], bv.y + sigma * acc[mt][h][2 * rr + 1]);
                        }
                    }
            }
            // The slot was only read here (ldmatrix, base loads), which the
            // barrier orders before the next copies; the zeroed padding of a
            // ragged rank is the one generic write the async copies must follow.
            if (r_ragged) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&W.empty[s]);
        }
    }
}

template <int TM, int RMAX>
__global__ void __launch_bounds__(kWideThreads, 1) lora_wide_expand_kernel(const __grid_constant__ WideParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        const WideBars W = wide_bars(k, smem);
        for (int i = 0; i < k.S; ++i) {
            mbar_init(&W.full[i], 1);
            mbar_init(&W.done[i], kWideConsumers);
            mbar_init(&W.empty[i], kWideConsumers);
        }
        fence_mbar_init();
        prefetch_tmap(&k.tmB);
        if (k.p.b_tuple)
            for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmBs[j]);
    }
    int nruns = 0;
    int *tables = reinterpret_cast<int *>(smem + k.o_run);
    const int ntiles = build_run_table_raw<TM>(k.p, k.max_segments, k.runcap, tables, &nruns);  // ends with __syncthreads
    const int ncols = k.p.off[k.p.c] - k.p.off[0];
    const int nblk = (ncols + k.cb - 1) / k.cb;
    const int units = ntiles * nblk;
    if (warp == 0) wide_load<TM>(k, smem, tables, nruns, nblk, units);
    else if (warp >= 2) wide_consume<TM, RMAX>(k, smem, tables, nruns, nblk, units, warp - 2);
}

}  // namespace

const void *lora_kernel_wide(int tm, int rmax) {
#define CSGMV_W(TM_, R_) \
    if (tm == TM_ && rmax == R_) return reinterpret_cast<const void *>(lora_wide_expand_kernel<TM_, R_>);
    CSGMV_W(16, 16) CSGMV_W(16, 32) CSGMV_W(16, 64) CSGMV_W(32, 16) CSGMV_W(32, 32) CSGMV_W(32, 64)
#undef CSGMV_W
    return nullptr;
}

}  // namespace csgmv
