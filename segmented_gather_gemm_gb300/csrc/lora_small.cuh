// Small-tile (16 / 32 token) kernel of the csgmv LoRA path, the decode shape
// (sglang chunked_backend.py run_qkv_lora / run_gate_up_lora,
// run_lora_a_sgemm, run_lora_b_sgemm; shapes from base_backend.py).
//
// A decode tile is a handful of tokens of one slot.  Per unit a cluster of CS
// CTAs splits K for the shrink and the output columns for the expand, like
// the 128-token cluster kernel, but every copy is a bulk copy, issued by many
// threads at once, so that the whole unit is in flight within a microsecond:
//   shrink  the CTA's whole K range in one shot: the slot's A rows as one
//           64-wide TMA box per K chunk (warp w issues chunks w, w+16, ...,
//           before the token list is even read) and each token's x row as
//           one contiguous bulk copy into a padded row-major tile; mma.sync
//           m16n8k16 with fp32 accumulators over all chunks;
//   reduce  partials summed over the cluster through distributed shared
//           memory: each CTA sums its share of the rows and writes the sums
//           into every CTA's copy of h, so the expand reads h locally (as
//           bf16 hi + lo fragment pairs);
//   expand  a ring of 256-column stages (512 in expand-only launches on
//           16-token tiles): the slot's B rows as TMA boxes of up to 256 rows
//           and each token's base row piece as one bulk copy; y = base +
//           sigma h B^T on the tensor cores in place, then 16-byte row stores.
// Every barrier arrival carries the bytes its thread copies (expect-tx), so
// one wait covers a whole stage.  All waits are bounded.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

struct SmallBars {
    uint64_t *x_full, *ex_full, *ex_empty;
};

__device__ __forceinline__ SmallBars small_bars(const TmaKernelParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    SmallBars r;
    r.x_full = b;
    r.ex_full = b + 1;
    r.ex_empty = b + 1 + k.S2;
    return r;
}

// Geometry of the small-tile kernel.  Expand stages are 256 columns wide, and
// 512 for expand-only launches on 16-token tiles: those stream long column
// ranges (a vocabulary-wide lm_head), where per-stage fixed costs dominate.
template <int TM, int MODE>
struct SmallGeo {
    static constexpr int WM = TM / 16;
    static constexpr int WN = kConsumerWarps / WM;
    static constexpr int NT = (TM == 16 && MODE == kModeExpand) ? 512 : 256;
    static constexpr int WCOLS = NT / WN;
    static constexpr int EXT = WCOLS / 8;
    static constexpr int BBOX = 256;  // rows of one B box (the TMA box limit)
};

template <int TM, int RMAX, int MODE>
__device__ void small_loop(const TmaKernelParams &k, unsigned char *smem, int q, int CS, int nruns,
                           int64_t nunits, int cid, int ncl) {
    using G = SmallGeo<TM, MODE>;
    constexpr int SHT = (3 * RMAX / 8 + G::WN - 1) / G::WN;  // shrink n8 tiles per warp (c <= 3)
    constexpr int KS = RMAX / 16;                             // expand k16 steps at most
    const LoraParams &p = k.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp / G::WN, wn = warp % G::WN;
    const SmallBars B = small_bars(k, smem);
    int *tok = reinterpret_cast<int *>(smem + k.o_tok);
    float *hpart = reinterpret_cast<float *>(smem + k.o_hpart);
    float *hfull = reinterpret_cast<float *>(smem + k.o_hred);  // [TM][hp] reduced h, every row
    unsigned char *xs = smem + k.o_sh;  // [TM][xpitch] x rows
    unsigned char *as = smem + k.o_ah;  // [kc_per][a_rows * 128] A boxes (128-byte swizzle)
    const int hp = k.hp;
    const int cR = p.c * p.R;
    const int nkc = (int)((p.K + 63) / 64);
    const int kc0 = (int)((int64_t)q * nkc / CS), kc1 = (int)((int64_t)(q + 1) * nkc / CS);
    const int nch = kc1 - kc0;
    const int64_t kend = (int64_t)kc1 * 64 < p.K ? (int64_t)kc1 * 64 : p.K;
    const int xcols = nch > 0 ? (int)(kend - (int64_t)kc0 * 64) : 0;
    const int rpr = TM / CS;  // rows of the reduction owned by each CTA
    const uint32_t abox = (uint32_t)k.a_rows * 128;
    uint32_t x_it = 0, ex_is = 0, ex_it = 0;

    for (int64_t u = cid; u < nunits; u += ncl) {
        const Unit U = decode_unit<TM>(k, smem, nruns, u);
        // token-list entry m_tok of this thread (the last warps read the list),
        // loaded alongside the slot's rank; p0 + m < num_tokens for m < M
        const int m_tok = kConsumerThreads - 1 - tid;
        const int t_pre = m_tok < TM && m_tok < U.M ? p.permutation[U.p0 + m_tok] : -1;
        const int r = unit_rank(p, U, q == 0 && tid == 0);
        if (r < 0) continue;
        int nt = 0, n0 = 0, n1 = 0;
        if constexpr (MODE != kModeShrink) {
            column_range(p, U.nb, q, CS, &n0, &n1);
            nt = n1 > n0 ? (n1 - n0 + G::NT - 1) / G::NT : 0;
        }
        if (r == 0) {
            // shrink: zero h rows; non-accumulating expand: zero output rows
            if constexpr (MODE == kModeShrink) {
                for (int m = q; m < U.M; m += CS) {
                    const int t = p.permutation[U.p0 + m];
                    if (t < 0 || t >= p.num_tokens) continue;
                    for (int col = tid; col < cR; col += kConsumerThreads) {
                        if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = 0.f;
                        else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(0.f);
                    }
                }
            } else if constexpr (MODE == kModeExpand) {
                if (!p.accumulate) {
                    const int nch8 = (n1 - n0) / 8;
                    for (int m = 0; m < U.M; ++m) {
                        const int t = p.permutation[U.p0 + m];
                        if (t < 0 || t >= p.num_tokens) continue;
                        for (int ch = tid; ch < nch8; ch += kConsumerThreads)
                            *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + n0 + 8 * ch) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            continue;
        }
        const float sigma = p.scalings[U.w];
        const int cr = p.c * r;
        const int crp = (cr + 7) & ~7;
        const int ksteps = (r + 15) / 16;

        fence_proxy_async_smem();  // this thread's generic writes before bulk copies reuse the memory
        __syncthreads();           // every warp is done with the previous unit's tiles and token list

        // The A boxes depend on the slot alone: out before the token list.
        uint32_t my_bytes = 0;
        if constexpr (MODE != kModeExpand) {
            if (lane == 0)
                for (int ci = warp; ci < nch; ci += kConsumerWarps) {
                    tma_load_2d(as + ci * abox, &k.tmA, (kc0 + ci) * 64, U.w * cR, B.x_full);
                    my_bytes += abox;
                }
        }
        // token list, written by the last warps (the first ones are issuing TMA)
        if (m_tok >= 0 && m_tok < TM) {
            int t = -1;
            if (m_tok < U.M) {
                t = t_pre;
                if (t < 0 || t >= p.num_tokens) {
                    atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
                    t = -1;
                }
            }
            tok[m_tok] = t;
        }
        __syncthreads();

        // Row copies are spread over the warps (row m: warp m % 16, lane m / 16),
        // since one warp issues its lanes' bulk copies one after another.
        const int my_row = lane < TM / kConsumerWarps ? lane * kConsumerWarps + warp : -1;
        if constexpr (MODE != kModeExpand) {
            // x rows: token m's K range [kc0*64, kc0*64 + xcols) in one bulk copy;
            // staged columns past K (a partial last chunk) are zero, since stale
            // values there could be NaN and meet the zero-filled A columns.
            const int t = my_row >= 0 && my_row < U.M ? tok[my_row] : -1;
            if (my_row >= 0) {
                __nv_bfloat16 *row = reinterpret_cast<__nv_bfloat16 *>(xs + my_row * k.xpitch);
                for (int col = xcols; col < nch * 64; ++col) row[col] = __float2bfloat16_rn(0.f);
                if (t >= 0 && xcols > 0) my_bytes += (uint32_t)xcols * 2;
            }
            mbar_arrive_expect_tx(B.x_full, my_bytes);
            if (t >= 0 && xcols > 0)
                bulk_g2s(xs + my_row * k.xpitch, p.x + (int64_t)t * p.K + (int64_t)kc0 * 64, (uint32_t)xcols * 2,
                         B.x_full);
        }

        // base rows and B rows of expand stage `i` into the next ring slot
        auto issue_stage = [&](int i) {
            const int e = ex_is % k.S2;
            mbar_wait(&B.ex_empty[e], ((ex_is / k.S2) & 1) ^ 1, p.status, kStatusTimeout);
            unsigned char *ys = smem + k.o_ex + e * k.ex_stage;
            const int x0 = n0 + i * G::NT, x1 = min(n1, x0 + G::NT);
            const int t = my_row >= 0 && my_row < U.M ? tok[my_row] : -1;
            const bool row_copy = t >= 0 && p.accumulate;
            const bool b_copy = tid == kConsumerThreads - 1;  // a lane of its own: the last warp's last
            uint32_t bytes = 0;
            if (b_copy) bytes += (uint32_t)G::NT * p.R * 2;
            if (row_copy) bytes += (uint32_t)(x1 - x0) * 2;
            mbar_arrive_expect_tx(&B.ex_full[e], bytes);
            if (b_copy)
                for (int bb = 0; bb < G::NT / G::BBOX; ++bb)
                    load_b_rows(k, ys + k.ex_b + bb * G::BBOX * p.R * 2, U.w, x0 + bb * G::BBOX, G::BBOX,
                                &B.ex_full[e]);
            if (row_copy)
                bulk_g2s(ys + my_row * k.ypitch, p.y + (int64_t)t * p.N + x0, (uint32_t)(x1 - x0) * 2, &B.ex_full[e]);
            ++ex_is;
        };
        const int ex_pre = min(nt, k.S2 - 1);
        for (int i = 0; i < ex_pre; ++i) issue_stage(i);

        if constexpr (MODE != kModeExpand) {
            // ---------------------------------------------------------------- shrink
            mbar_wait(B.x_full, x_it & 1, p.status, kStatusTimeout);
            ++x_it;
            // Two accumulator sets (even / odd k16 steps); per chunk every
            // fragment is loaded before the MMAs, so the loads overlap.
            float acc[2][SHT][4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int i = 0; i < SHT; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[h2][i][e] = 0.f;
            const unsigned char *xrow = xs + (wm * 16 + (lane & 15)) * k.xpitch + 16 * (lane >> 4);
            for (int ci = 0; ci < nch; ++ci) {
                const __nv_bfloat16 *ab = reinterpret_cast<const __nv_bfloat16 *>(as + ci * abox);
                uint32_t a[4][4], b[4][SHT][2];
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    ldmatrix_x4(a[ks][0], a[ks][1], a[ks][2], a[ks][3], xrow + (ci * 64 + ks * 16) * 2);
#pragma unroll
                    for (int i = 0; i < SHT; ++i) {
                        const int j = wn + G::WN * i;
                        if (j * 8 < crp)
                            ldmatrix_x2(b[ks][i][0], b[ks][i][1],
                                        ab + swz(j * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1), 8, 0));
                    }
                }
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                    for (int i = 0; i < SHT; ++i)
                        if ((wn + G::WN * i) * 8 < crp) mma_bf16_16816(acc[ks & 1][i], a[ks], b[ks][i][0], b[ks][i][1]);
            }
#pragma unroll
            for (int i = 0; i < SHT; ++i) {
                const int j = wn + G::WN * i;
                if (j * 8 < crp) {
                    float v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = acc[0][i][e] + acc[1][i][e];
                    const int row = wm * 16 + (lane >> 2), col = j * 8 + 2 * (lane & 3);
                    *reinterpret_cast<float2 *>(hpart + row * hp + col) = make_float2(v[0], v[1]);
                    *reinterpret_cast<float2 *>(hpart + (row + 8) * hp + col) = make_float2(v[2], v[3]);
                }
            }
            // ---------------------------------------------------------------- reduce
            if (CS > 1) {
                cluster_arrive();
                cluster_wait();
                const int nv = crp >> 2;
                for (int idx = tid; idx < rpr * nv; idx += kConsumerThreads) {
                    const int rr = idx / nv, v = idx % nv;
                    const int row = q * rpr + rr;
                    if (row >= U.M) continue;
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int p0 = 0; p0 < CS; p0 += 8) {  // clusters of up to 16 CTAs
                        // eight peers' partials are loaded before any is summed
                        float4 t4[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            if (p0 + jj < CS) t4[jj] = dsmem_ld_f4(dsmem_addr(hpart + row * hp + 4 * v, p0 + jj));
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            if (p0 + jj < CS) {
                                s4.x += t4[jj].x; s4.y += t4[jj].y; s4.z += t4[jj].z; s4.w += t4[jj].w;
                            }
                    }
                    for (int peer = 0; peer < CS; ++peer)
                        dsmem_st_f4(dsmem_addr(hfull + row * hp + 4 * v, peer), s4);
                }
                cluster_arrive();  // every CTA's hfull is complete after this barrier
                cluster_wait();
            } else {
                named_bar_sync(kBarConsumers, kConsumerThreads);
            }
            if constexpr (MODE == kModeShrink) {
                const float *src = CS > 1 ? hfull : hpart;
                const int row0 = CS > 1 ? q * rpr : 0;
                const int nrows = CS > 1 ? rpr : TM;
                for (int idx = tid; idx < nrows * cR; idx += kConsumerThreads) {
                    const int rr = idx / cR, col = idx % cR;
                    const int row = row0 + rr;
                    if (row >= U.M) continue;
                    const int t = tok[row];
                    if (t < 0) continue;
                    const float v = col < cr ? src[row * hp + col] : 0.f;
                    if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = v;
                    else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(v);
                }
            }
        }

        if constexpr (MODE != kModeShrink) {
            // ---------------------------------------------------------------- expand
            const int rowA = wm * 16 + (lane >> 2), rowB = rowA + 8;
            uint32_t fhi[KS][4], flo[KS][4];
            int cur = -1;
            auto h_at = [&](int row, int col) -> float {  // h[row][col], 0 beyond the tile
                if (row >= U.M) return 0.f;
                if constexpr (MODE == kModeExpand) {
                    const int t = tok[row];
                    if (t < 0) return 0.f;
                    if (p.h_f32) return reinterpret_cast<const float *>(p.h)[(int64_t)t * p.ldh + col];
                    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col]);
                } else {
                    return (CS > 1 ? hfull : hpart)[row * hp + col];
                }
            };
            auto load_slice = [&](int j) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int k0 = ks * 16 + 2 * (lane & 3);
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int kk = k0 + (e & 1) + ((e & 4) ? 8 : 0);
                        const int row = (e & 2) ? rowB : rowA;
                        v[e] = kk < r ? h_at(row, j * r + kk) : 0.f;
                    }
                    split_pair(v[0], v[1], fhi[ks][0], flo[ks][0]);
                    split_pair(v[2], v[3], fhi[ks][1], flo[ks][1]);
                    split_pair(v[4], v[5], fhi[ks][2], flo[ks][2]);
                    split_pair(v[6], v[7], fhi[ks][3], flo[ks][3]);
                }
                cur = j;
            };
            // B tile: row n holds B[w][x0 + n][0:R], R*2 bytes, swizzled like the TMA box
            const int pcB = p.R / 8, shB = pc_shift_of(pcB);
            const bool r_ragged = p.R == 8 ? (r < 8) : (r % 16 != 0);
            // h of the first slice this warp needs, pulled while stage 0 lands
            if (nt > 0) {
                const int wc = n0 + wn * G::WCOLS;
                if (wc < min(n1, n0 + G::NT)) load_slice(slice_at(p, wc));
            }
            for (int i = 0; i < nt; ++i) {
                if (i + k.S2 - 1 < nt) issue_stage(i + k.S2 - 1);
                const int e = ex_it % k.S2;
                mbar_wait(&B.ex_full[e], (ex_it / k.S2) & 1, p.status, kStatusTimeout);
                unsigned char *ys = smem + k.o_ex + e * k.ex_stage;
                const __nv_bfloat16 *bs = reinterpret_cast<const __nv_bfloat16 *>(ys + k.ex_b);
                const int x0 = n0 + i * G::NT, x1 = min(n1, x0 + G::NT);
                if (r_ragged) {
                    // B columns [r, 16*ceil(r/16)) are adapter padding: zero them
                    // so that padding never reaches the output (even NaN).
                    const int rpad = p.R == 8 ? 8 : (r + 15) / 16 * 16;
                    const int npad = rpad - r;
                    __nv_bfloat16 *bw = const_cast<__nv_bfloat16 *>(bs);
                    for (int idx = tid; idx < G::NT * npad; idx += kConsumerThreads) {
                        const int n = idx / npad, kk = r + idx % npad;
                        bw[swz(n, kk >> 3, pcB, shB) + (kk & 7)] = __float2bfloat16_rn(0.f);
                    }
                    named_bar_sync(kBarConsumers, kConsumerThreads);
                }
                float acc[G::EXT][4];
#pragma unroll
                for (int t8 = 0; t8 < G::EXT; ++t8)
#pragma unroll
                    for (int ee = 0; ee < 4; ++ee) acc[t8][ee] = 0.f;
                const int wc0 = x0 + wn * G::WCOLS;  // first column of this warp
                if (wc0 < x1) {
                    const int jl = slice_at(p, wc0), jh = slice_at(p, min(wc0 + G::WCOLS, x1) - 1);
                    for (int jj = jl; jj <= jh; ++jj) {
                        if (jj != cur) load_slice(jj);
#pragma unroll
                        for (int t8 = 0; t8 < G::EXT; t8 += 2) {
                            const int lc = wn * G::WCOLS + 8 * t8;
                            if (x0 + lc >= x1) continue;
                            const bool use0 = jl == jh || slice_at(p, x0 + lc) == jj;
                            const bool use1 = x0 + lc + 8 < x1 && (jl == jh || slice_at(p, x0 + lc + 8) == jj);
                            // every B fragment of the pair first, then the MMAs
                            uint32_t bf[KS][4];
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks) {
                                if (ks < ksteps) {
                                    if (RMAX == 16 && p.R == 8) {
                                        const int nrow = lc + 8 * ((lane >> 3) & 1) + (lane & 7);
                                        ldmatrix_x2(bf[ks][0], bf[ks][2], bs + nrow * 8);
                                        bf[ks][1] = 0u;
                                        bf[ks][3] = 0u;
                                    } else {
                                        const int nrow = lc + 8 * (lane >> 4) + (lane & 7);
                                        const int ch = 2 * ks + ((lane >> 3) & 1);
                                        ldmatrix_x4(bf[ks][0], bf[ks][1], bf[ks][2], bf[ks][3], bs + swz(nrow, ch, pcB, shB));
                                    }
                                }
                            }
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks) {
                                if (ks < ksteps) {
                                    if (use0) {
                                        mma_bf16_16816(acc[t8], fhi[ks], bf[ks][0], bf[ks][1]);
                                        mma_bf16_16816(acc[t8], flo[ks], bf[ks][0], bf[ks][1]);
                                    }
                                    if (use1) {
                                        mma_bf16_16816(acc[t8 + 1], fhi[ks], bf[ks][2], bf[ks][3]);
                                        mma_bf16_16816(acc[t8 + 1], flo[ks], bf[ks][2], bf[ks][3]);
                                    }
                                }
                            }
                        }
                    }
                }
                // y = base + sigma * acc into this warp's scratch tile (the staged
                // base rows are only read, so the next bulk copy into the stage
                // needs no proxy fence)
                constexpr int SP = G::WCOLS * 2 + 16;  // scratch row pitch, bytes
                unsigned char *wsc = smem + k.o_hpart + k.wscr_off + warp * 16 * SP;
#pragma unroll
                for (int t8 = 0; t8 < G::EXT; ++t8) {
                    const int lc = wn * G::WCOLS + 8 * t8 + 2 * (lane & 3);
                    if (x0 + wn * G::WCOLS + 8 * t8 >= x1) continue;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int row = hh ? rowB : rowA;
                        const float2 bv = p.accumulate && row < U.M
                                              ? unpack_bf16x2(*reinterpret_cast<const uint32_t *>(ys + row * k.ypitch + lc * 2))
                                              : make_float2(0.f, 0.f);
                        *reinterpret_cast<uint32_t *>(wsc + (row - wm * 16) * SP + (lc - wn * G::WCOLS) * 2) =
                            pack_bf16x2(bv.x + sigma * acc[t8][2 * hh], bv.y + sigma * acc[t8][2 * hh + 1]);
                    }
                }
                __syncwarp();
                // this warp's 16 rows x WCOLS columns go out as 16-byte stores
                constexpr int CPR = G::WCOLS / 8;  // 16-byte chunks per row
                for (int idx = lane; idx < 16 * CPR; idx += 32) {
                    const int rr = idx / CPR, c16 = idx % CPR;
                    const int row = wm * 16 + rr;
                    const int col = x0 + wn * G::WCOLS + 8 * c16;
                    if (row >= U.M || col >= x1) continue;
                    const int t = tok[row];
                    if (t < 0) continue;
                    *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) =
                        *reinterpret_cast<const uint4 *>(wsc + rr * SP + c16 * 16);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.ex_empty[e]);
                ++ex_it;
            }
        }
    }
}

template <int TM, int RMAX, int MODE>
__global__ void __launch_bounds__(kConsumerThreads, 1) lora_small_kernel(const __grid_constant__ TmaKernelParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment of the dynamic window for the 128-byte swizzle
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    int CS = 1, q = 0;
    if constexpr (MODE != kModeExpand) {
        CS = (int)cluster_size();
        q = (int)cluster_rank();
    }
    if (threadIdx.x == 0) {
        const SmallBars B = small_bars(k, smem);
        mbar_init(B.x_full, kConsumerThreads);
        for (int i = 0; i < k.S2; ++i) {
            mbar_init(&B.ex_full[i], kConsumerThreads);
            mbar_init(&B.ex_empty[i], kConsumerWarps);
        }
        fence_mbar_init();
        prefetch_tmap(&k.tmA);
        prefetch_tmap(&k.tmB);
        if (k.p.b_tuple)
            for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmBs[j]);
    }
    int nruns = 0;
    const int ntiles = build_run_table<TM>(k, smem, &nruns);  // ends with __syncthreads
    const int64_t nunits = (int64_t)ntiles * k.p.nsplit;
    const int cid = blockIdx.x / CS, ncl = gridDim.x / CS;
    small_loop<TM, RMAX, MODE>(k, smem, q, CS, nruns, nunits, cid, ncl);
    if constexpr (MODE != kModeExpand) {
        if (CS > 1) {  // peers may still read this CTA's shared memory
            cluster_arrive();
            cluster_wait();
        }
    }
}

}  // namespace csgmv
