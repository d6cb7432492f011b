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

// Grouped table (ints from `g`): cnt[nslot] tokens per slot, base[nslot + 1]
// first list entry per slot, tile0[nslot + 1] first tile per slot,
// scnt[nslot] segments per slot (then running ranks), sbase[nslot + 1] first
// sorted segment per slot, wseg / ia / ib[segcap] slot, first and end
// position of each segment, srt[segcap] segments sorted by slot (stable),
// list[tokcap] positions slot by slot, scratch[32].  Every CTA builds the
// table alone, so its order must not depend on timing: segments are ranked
// within their slot by index, and no atomic decides a place.
struct WGroup {
    int *cnt, *base, *tile0, *scnt, *sbase, *wseg, *ia, *ib, *srt, *list, *scratch;
};

__device__ __forceinline__ WGroup wide_group(const WideParams &k, int *g) {
    WGroup G;
    G.cnt = g;
    G.base = G.cnt + k.nslot;
    G.tile0 = G.base + k.nslot + 1;
    G.scnt = G.tile0 + k.nslot + 1;
    G.sbase = G.scnt + k.nslot;
    G.wseg = G.sbase + k.nslot + 1;
    G.ia = G.wseg + k.segcap;
    G.ib = G.ia + k.segcap;
    G.srt = G.ib + k.segcap;
    G.list = G.srt + k.segcap;
    G.scratch = G.list + k.tokcap;
    return G;
}

// Builds the grouped table; returns the tile count.  Every thread of the
// block calls it, and it ends with a block barrier.  A slot id out of range
// is reported and its tokens are left out (their rows stay as they are, as
// on every other path); more positions than tokcap (overlapping segments) are
// reported and give no tiles.
template <int TM>
__device__ int wide_group_table(const WideParams &k, int *g) {
    const LoraParams &p = k.p;
    const WGroup G = wide_group(k, g);
    const int tid = threadIdx.x, nt = blockDim.x, L = k.nslot, lane = tid & 31;
    griddep_wait();  // the batch info may come from the kernel launched just before
    for (int i = tid; i < L; i += nt) {
        G.cnt[i] = 0;
        G.scnt[i] = 0;
    }
    const int nseg = max(0, min(*p.num_segments_dev, min(k.max_segments, k.segcap)));
    __syncthreads();
    // slot and bounds of every segment; tokens and segments per slot
    for (int s = tid; s < nseg; s += nt) {
        int w = p.weight_indices[s];
        const int a = max(0, min(p.seg_indptr[s], p.num_tokens)), b = max(a, min(p.seg_indptr[s + 1], p.num_tokens));
        if (w < 0 || w >= L) {
            if (b > a) atomicOr(p.status, CSGMV_STATUS_BAD_ADAPTER);
            w = -1;
        } else {
            atomicAdd(&G.cnt[w], b - a);
            atomicAdd(&G.scnt[w], 1);
        }
        G.wseg[s] = w;
        G.ia[s] = a;
        G.ib[s] = b;
    }
    __syncthreads();
    int pcarry = 0, tcarry = 0, scarry = 0;
    for (int w0 = 0; w0 < L; w0 += nt) {
        const int w = w0 + tid;
        const int c = w < L ? G.cnt[w] : 0, sc = w < L ? G.scnt[w] : 0;
        int ptot, ttot, stot;
        const int ppre = block_scan(c, G.scratch, &ptot);
        const int tpre = block_scan((c + TM - 1) / TM, G.scratch, &ttot);
        const int spre = block_scan(sc, G.scratch, &stot);
        if (w < L) {
            G.base[w] = pcarry + ppre;
            G.tile0[w] = tcarry + tpre;
            G.sbase[w] = scarry + spre;
        }
        pcarry += ptot;
        tcarry += ttot;
        scarry += stot;
    }
    const bool fits = pcarry <= k.tokcap;
    if (tid == 0) {
        G.base[L] = pcarry;
        G.tile0[L] = tcarry;
        G.sbase[L] = scarry;
        if (!fits) atomicOr(p.status, CSGMV_STATUS_CAPACITY);
    }
    for (int i = tid; i < L; i += nt) G.scnt[i] = 0;
    __syncthreads();
    if (!fits) return 0;
    // rank of each segment among the earlier segments of its slot, one warp
    // over batches of 32 segments in order: lanes on one slot are matched,
    // ranked by lane, and the group's last lane moves the slot's count on
    if (tid < 32) {
        for (int s0 = 0; s0 < nseg; s0 += 32) {
            const int s = s0 + lane;
            const int w = s < nseg ? G.wseg[s] : -1;
            const unsigned m = __match_any_sync(0xffffffffu, w);
            const int before = w >= 0 ? G.scnt[w] : 0;
            __syncwarp();
            if (w >= 0) {
                G.srt[G.sbase[w] + before + __popc(m & ((1u << lane) - 1u))] = s;
                if (lane == 31 - __clz((int)m)) G.scnt[w] = before + __popc(m);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // positions in sorted-segment order: slot w's tokens fill
    // [base[w], base[w + 1]) in segment order
    int ocarry = 0;
    for (int i0 = 0; i0 < scarry; i0 += nt) {
        const int i = i0 + tid;
        const int sg = i < scarry ? G.srt[i] : 0;
        const int a = i < scarry ? G.ia[sg] : 0, n = i < scarry ? G.ib[sg] - a : 0;
        int tot;
        const int o = ocarry + block_scan(n, G.scratch, &tot);
        for (int e = 0; e < n; ++e) G.list[o + e] = a + e;
        ocarry += tot;
    }
    __syncthreads();
    return tcarry;
}

template <int TM>
__device__ __forceinline__ bool wide_unit(const WideParams &k, const int *tables, int nruns, int nblk, int u,
                                          bool report, WUnit &U) {
    const LoraParams &p = k.p;
    Unit T;
    if (nruns < 0) {  // grouped table
        // slot: the last with tile0 <= tile (slots without tokens end below it)
        const WGroup G = wide_group(k, const_cast<int *>(tables));
        const int tile = u / nblk;
        int lo = 0, hi = k.nslot;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (G.tile0[mid] <= tile) lo = mid; else hi = mid;
        }
        T.w = lo;
        T.p0 = G.base[lo] + (tile - G.tile0[lo]) * TM;  // list entry of row 0
        T.M = min(TM, G.base[lo + 1] - T.p0);
        T.nb = 0;
    } else {
        T = tile_of<TM>(tables, k.runcap, nruns, u / nblk);
    }
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
__device__ __forceinline__ int wide_token(const WideParams &k, const int *tables, int nruns, const WUnit &U, int row) {
    const LoraParams &p = k.p;
    if (row >= U.M) return -1;
    const int pos = nruns < 0 ? wide_group(k, const_cast<int *>(tables)).list[U.p0 + row] : U.p0 + row;
    const int t = p.permutation[pos];
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
        const int t = lane < TM ? wide_token(k, tables, nruns, U, lane) : -1;
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

// ----------------------------------------------------------------------------------------- h prep
// The spare warp, for one-slice outputs: per unit (the consumers' order) the
// tokens of its TM = 16 rows and the h fragments every consumer lane holds
// (lane L: rows L / 4 and L / 4 + 8, columns 2 (L % 4) + {0, 1, 8, 9} of each
// k16 step, planes summed in part order), as bf16 hi / lo pairs, into buffer
// it % 2 once the consumers have taken what it held before.
template <int TM, int RMAX>
__device__ void wide_hprep(const WideParams &k, unsigned char *smem, const int *tables, int nruns, int nblk,
                           int units) {
    constexpr int KS = RMAX / 16;
    static_assert(TM == 16, "one 16-row tile per unit");
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    uint64_t *hfull = reinterpret_cast<uint64_t *>(smem + k.o_hbar), *hempty = hfull + 2;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        WUnit U;
        if (!wide_unit<TM>(k, tables, nruns, nblk, u, false, U)) continue;
        const int b = it & 1;
        mbar_wait(&hempty[b], ((it >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        uint32_t *hf = reinterpret_cast<uint32_t *>(smem + k.o_hf) + b * kWideHfInts;
        int *tok = reinterpret_cast<int *>(smem + k.o_hf) + 2 * kWideHfInts + b * 32;
        const int t = lane < TM ? wide_token(k, tables, nruns, U, lane) : -1;
        tok[lane] = t;
        const int tA = __shfl_sync(0xffffffffu, t, lane >> 2), tB = __shfl_sync(0xffffffffu, t, (lane >> 2) + 8);
        float v[KS][8];
        const int parts = max(1, p.h_parts);
#pragma unroll
        for (int q = 0; q < kMaxKParts; ++q) {
            if (q > 0 && q >= parts) break;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int kk = ks * 16 + 2 * (lane & 3) + (e & 1) + ((e & 4) ? 8 : 0);
                    const int tt = (e & 2) ? tB : tA;
                    float x = 0.f;
                    if (kk < U.r && tt >= 0) {
                        const int64_t o = (int64_t)q * p.h_plane + (int64_t)tt * p.ldh + kk;
                        x = p.h_f32 ? reinterpret_cast<const float *>(p.h)[o]
                                    : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[o]);
                    }
                    v[ks][e] = q == 0 ? x : v[ks][e] + x;
                }
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int rg = 0; rg < 4; ++rg) {
                uint32_t hi, lo;
                split_pair(v[ks][2 * rg], v[ks][2 * rg + 1], hi, lo);
                hf[((ks * 2 + 0) * 4 + rg) * 32 + lane] = hi;
                hf[((ks * 2 + 1) * 4 + rg) * 32 + lane] = lo;
            }
        mbar_arrive(&hfull[b]);  // every lane: its own writes are released
        ++it;
    }
}

// --------------------------------------------------------------------------------------- consume
// NT8 = n8 tiles per consumer warp and stage (k.nt / kWideConsumers / 8).
// In the one-slice path the warp's n8 tile j, row n holds stage column
// lc0 + 2 * NT8 * (n / 2) + 2 * j + n % 2: the accumulator layout of
// m16n8k16 (lane holds columns 2 (lane % 4) + {0, 1} of each n8 tile) then
// gives lane q = lane % 4 the 2 * NT8 consecutive columns lc0 + 2 NT8 q + ...
template <int TM, int RMAX, int NT8>
__device__ void wide_consume(const WideParams &k, unsigned char *smem, const int *tables, int nruns, int nblk,
                             int units, int cw) {
    constexpr int KS = RMAX / 16, NMT = TM / 16;
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const WideBars W = wide_bars(k, smem);
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    const int wcols = 8 * NT8;  // this warp's columns of a stage: [lc0, lc0 + wcols)
    const int lc0 = cw * wcols;
    const bool R8 = RMAX == 16 && p.R == 8;
    const int cq = lc0 + 2 * NT8 * (lane & 3);  // first stage column of this lane's piece
    // per-lane ldmatrix offsets (bytes into a stage's B rows) of the permuted
    // rows: matrix pair qq covers n8 tiles 2 qq, 2 qq + 1
    uint32_t boff[NT8 / 2][KS];
#pragma unroll
    for (int qq = 0; qq < NT8 / 2; ++qq)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int n = lane & 7;
            if (R8) {
                const int j = 2 * qq + ((lane >> 3) & 1);
                boff[qq][ks] = (uint32_t)(lc0 + 2 * NT8 * (n >> 1) + 2 * j + (n & 1)) * 16u;
            } else {
                const int j = 2 * qq + (lane >> 4);
                const int row = lc0 + 2 * NT8 * (n >> 1) + 2 * j + (n & 1);
                boff[qq][ks] = (uint32_t)swz(row, 2 * ks + ((lane >> 3) & 1), pcB, shB) * 2u;
            }
        }
    // the spare warp prepares h for one-slice outputs (TM = 16 only)
    const bool hprep = TM == 16 && p.c == 1;
    uint64_t *hfull = reinterpret_cast<uint64_t *>(smem + k.o_hbar), *hempty = hfull + 2;
    uint32_t it = 0, hit = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        WUnit U;
        if (!wide_unit<TM>(k, tables, nruns, nblk, u, false, U)) continue;
        const float sigma = U.r > 0 ? p.scalings[U.w] : 0.f;
        const int ksteps = (U.r + 15) / 16;
        const bool r_ragged = U.r > 0 && (p.R == 8 ? (U.r < 8) : (U.r % 16 != 0));
        // tokens of the rows this lane's fragments hold: mt * 16 + lane / 4 (+ 8),
        // and h of one slice as bf16 hi / lo A fragments, every 16-row tile
        int trow[NMT][2];
        uint32_t fhi[NMT][KS][4], flo[NMT][KS][4];
        int cur = -1;
        if (hprep) {  // one slice, 16-row tiles: from the spare warp
            const int b = hit & 1;
            mbar_wait(&hfull[b], (hit >> 1) & 1, p.status, kStatusTimeout);
            const uint32_t *hf = reinterpret_cast<const uint32_t *>(smem + k.o_hf) + b * kWideHfInts;
            const int *tok = reinterpret_cast<const int *>(smem + k.o_hf) + 2 * kWideHfInts + b * 32;
            trow[0][0] = tok[lane >> 2];
            trow[0][1] = tok[(lane >> 2) + 8];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int rg = 0; rg < 4; ++rg) {
                    fhi[0][ks][rg] = hf[((ks * 2 + 0) * 4 + rg) * 32 + lane];
                    flo[0][ks][rg] = hf[((ks * 2 + 1) * 4 + rg) * 32 + lane];
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hempty[b]);
            ++hit;
            cur = 0;
        } else {
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    trow[mt][hh] = wide_token(k, tables, nruns, U, mt * 16 + (lane >> 2) + 8 * hh);
        }
        auto load_slice = [&](int j) {
            // plane 0 of every value first (all loads in flight at once),
            // then the further planes in part order
            float v[NMT][KS][8];
            const int parts = max(1, p.h_parts);
#pragma unroll
            for (int q = 0; q < kMaxKParts; ++q) {
                if (q > 0 && q >= parts) break;
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int kk = ks * 16 + 2 * (lane & 3) + (e & 1) + ((e & 4) ? 8 : 0);
                            const int t = trow[mt][(e >> 1) & 1];
                            float x = 0.f;
                            if (kk < U.r && t >= 0) {
                                const int64_t o = (int64_t)q * p.h_plane + (int64_t)t * p.ldh + j * U.r + kk;
                                x = p.h_f32 ? reinterpret_cast<const float *>(p.h)[o]
                                            : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[o]);
                            }
                            v[mt][ks][e] = q == 0 ? x : v[mt][ks][e] + x;
                        }
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
            const uint32_t bs_u = smem_u32(bs), ys_u = smem_u32(ys);
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
                // one slice (always so for one output projection): NT8 n8 tiles
                // whose B rows are permuted so that each lane ends up with 2 * NT8
                // consecutive columns of its rows; every MMA first, then one
                // vector load of base and one vector store of y per row
                float acc[NT8][NMT][4];
#pragma unroll
                for (int j = 0; j < NT8; ++j)
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[j][mt][e] = 0.f;
                if (U.r > 0) {
                    const int jsl = slice_of_col(lcs);
                    if (jsl != cur) load_slice(jsl);
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        if (ks < ksteps) {
                            uint32_t bf[NT8][2];
#pragma unroll
                            for (int qq = 0; qq < NT8 / 2; ++qq) {
                                if (R8) {
                                    ldsm_x2(bf[2 * qq][0], bf[2 * qq + 1][0], bs_u + boff[qq][ks]);
                                    bf[2 * qq][1] = 0u;
                                    bf[2 * qq + 1][1] = 0u;
                                } else {
                                    uint32_t r4[4];
                                    ldsm_x4(r4, bs_u + boff[qq][ks]);
                                    bf[2 * qq][0] = r4[0];
                                    bf[2 * qq][1] = r4[1];
                                    bf[2 * qq + 1][0] = r4[2];
                                    bf[2 * qq + 1][1] = r4[3];
                                }
                            }
#pragma unroll
                            for (int j = 0; j < NT8; ++j)
#pragma unroll
                                for (int mt = 0; mt < NMT; ++mt) {
                                    mma_bf16_16816(acc[j][mt], fhi[mt][ks], bf[j][0], bf[j][1]);
                                    mma_bf16_16816(acc[j][mt], flo[mt][ks], bf[j][0], bf[j][1]);
                                }
                        }
                    }
                }
                // y = base + sigma * acc: this lane's 2 * NT8 columns cq .. of each
                // of its rows (stage lengths are multiples of 8 columns, so the
                // piece lies wholly inside or outside the stage)
                if (c0 + cq < c1) {
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int t = trow[mt][rr];
                            if (t < 0) continue;
                            const uint32_t ya = ys_u + (uint32_t)((mt * 16 + (lane >> 2) + 8 * rr) * k.ypitch + cq * 2);
                            uint32_t o[NT8];
                            if (NT8 == 4) {
                                const uint4 b = p.accumulate ? lds_v4(ya) : make_uint4(0u, 0u, 0u, 0u);
                                const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                                for (int j = 0; j < NT8; ++j) {
                                    const float2 f = unpack_bf16x2(bw[j]);
                                    o[j] = pack_bf16x2(f.x + sigma * acc[j][mt][2 * rr], f.y + sigma * acc[j][mt][2 * rr + 1]);
                                }
                                *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + c0 + cq) = make_uint4(o[0], o[1], o[2], o[3]);
                            } else {
                                const uint2 b = p.accumulate ? lds_v2(ya) : make_uint2(0u, 0u);
                                const uint32_t bw[2] = {b.x, b.y};
#pragma unroll
                                for (int j = 0; j < NT8; ++j) {
                                    const float2 f = unpack_bf16x2(bw[j]);
                                    o[j] = pack_bf16x2(f.x + sigma * acc[j][mt][2 * rr], f.y + sigma * acc[j][mt][2 * rr + 1]);
                                }
                                *reinterpret_cast<uint2 *>(p.y + (int64_t)t * p.N + c0 + cq) = make_uint2(o[0], o[1]);
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
        uint64_t *hb = reinterpret_cast<uint64_t *>(smem + k.o_hbar);
        mbar_init(&hb[0], 32);  // hfull: every lane of the h warp
        mbar_init(&hb[1], 32);
        mbar_init(&hb[2], kWideConsumers);  // hempty: one lane per consumer warp
        mbar_init(&hb[3], kWideConsumers);
        fence_mbar_init();
        prefetch_tmap(&k.tmB);
        if (k.p.b_tuple)
            for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmBs[j]);
    }
    int nruns = -1;  // -1: the grouped table
    int *tables = reinterpret_cast<int *>(smem + k.o_run);
    // A batch info the csgmv builder made (its tile table holds a count) has
    // each slot's tokens in one run already: runs are the groups.
    bool grouped = k.grouped;
    if (grouped && k.p.tile_table) {
        griddep_wait();  // the batch info may come from the kernel launched just before
        grouped = k.p.tile_table[0] < 0;
    }
    const int ntiles = grouped ? wide_group_table<TM>(k, tables)  // both end with __syncthreads
                               : build_run_table_raw<TM>(k.p, k.max_segments, k.runcap, tables, &nruns);
    const int ncols = k.p.off[k.p.c] - k.p.off[0];
    const int nblk = (ncols + k.cb - 1) / k.cb;
    const int units = ntiles * nblk;
    if (warp == 0) wide_load<TM>(k, smem, tables, nruns, nblk, units);
    else if (warp == 1) {
        if (TM == 16 && k.p.c == 1) wide_hprep<TM, RMAX>(k, smem, tables, nruns, nblk, units);
    }
    else if (warp >= 2) {
        if (k.nt == 512) wide_consume<TM, RMAX, 4>(k, smem, tables, nruns, nblk, units, warp - 2);
        else wide_consume<TM, RMAX, 2>(k, smem, tables, nruns, nblk, units, warp - 2);
    }
}

}  // namespace

const void *lora_kernel_wide(int tm, int rmax) {
#define CSGMV_W(TM_, R_) \
    if (tm == TM_ && rmax == R_) return reinterpret_cast<const void *>(lora_wide_expand_kernel<TM_, R_>);
    CSGMV_W(16, 16) CSGMV_W(16, 32) CSGMV_W(16, 64)
#undef CSGMV_W
    return nullptr;
}

}  // namespace csgmv
