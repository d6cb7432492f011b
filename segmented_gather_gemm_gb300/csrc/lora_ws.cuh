// Warp-specialized tcgen05 kernel of the csgmv LoRA path for 128-token tiles
// (prefill), in fused, shrink-only and expand-only modes (sglang
// chunked_backend.py run_qkv_lora / run_gate_up_lora, run_lora_a_sgemm,
// run_lora_b_sgemm; shapes from base_backend.py).
//
// One CTA per SM walks its units (128-token tile of one slot x a block of
// output columns).  The roles run concurrently, linked by mbarriers, and the
// shrink of the next unit streams while the expand of the current one does:
//   warp 0      shrink producer: the tile's token list, then x rows and the
//               slot's A tile per 64-wide K chunk into the shrink ring (x of a
//               tile of non-consecutive tokens by TMA 4-row gathers);
//   warp 1      expand producer: base rows and the slot's B tile per
//               64-column stage into the expand ring.  Tiles of consecutive
//               tokens load rows as TMA boxes; others gather rows with
//               16-byte cp.async.  Producers run ahead into later units,
//               bounded only by their rings;
//   warp 2      shrink MMA issuer (one lane): h = x A^T into a TMEM
//               accumulator over the whole K;
//   warp 3      expand MMA issuer (one lane): per stage y_delta = h B^T (h as
//               a bf16 hi + lo pair, so h keeps ~16 bits) into one of two TMEM
//               accumulators; completions free ring stages (tcgen05.commit);
//   warps 4..11 epilogue: h from TMEM into the bf16 hi / lo operand tiles
//               (or to global memory in shrink-only mode), then per stage the
//               accumulator from TMEM, base + sigma * delta in place in the
//               staged tile, and the tile back to global memory (one TMA box
//               store for a full tile of consecutive tokens, 16-byte stores
//               through the permutation otherwise).
// Every wait is bounded; on a timeout the kernel sets a status bit and ends.
//
// The launcher routes shrink-only calls here.  For fused and expand calls the
// cluster kernel (lora_tma.cuh) measured faster on the prefill shapes: with
// 64-column stages, the single MMA-issuing warp and the epilogue spend about a
// microsecond of barrier and issue latency per stage, and shared memory does
// not leave room for wider stages next to the h operand tiles.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kWsWarps = 12;
constexpr int kWsThreads = kWsWarps * 32;
constexpr int kWsEpiWarps = 8;
constexpr int kWsCols = 64;           // output columns per expand load stage
constexpr int kWsPairCols = 128;      // columns per MMA / epilogue step: a pair of load stages
constexpr int kWsTmemCols = 512;      // h accumulator [0, 256), two step accumulators [256, 512)
constexpr int kWsAccCol = 256;
constexpr int kWsBaseBytes = 128 * 128;  // one 128-row x 64-column bf16 base tile
constexpr int kWsEpiBar = 2;          // named barrier of the epilogue warps

struct WsBars {
    uint64_t *sh_full, *sh_empty, *ex_full, *ex_empty, *b_full;
    uint64_t *hacc_full, *hacc_empty, *ah_full, *ah_empty;
    uint64_t *acc_full, *acc_empty, *tok_full, *tok_empty;  // [2] each
    uint32_t *tmem_slot;
    int *tok;    // [2][128]
    int *flag;   // [2]: the tile's rows are consecutive tokens
};

__device__ __forceinline__ WsBars ws_bars(const TmaKernelParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    WsBars w;
    w.sh_full = b;
    w.sh_empty = b + k.S1;
    w.ex_full = b + 2 * k.S1;
    w.ex_empty = b + 2 * k.S1 + k.S2;
    w.b_full = b + 2 * k.S1 + 2 * k.S2;
    uint64_t *x = b + 2 * k.S1 + 3 * k.S2;
    w.hacc_full = x;
    w.hacc_empty = x + 1;
    w.ah_full = x + 2;
    w.ah_empty = x + 3;
    w.acc_full = x + 4;
    w.acc_empty = x + 6;
    w.tok_full = x + 8;
    w.tok_empty = x + 10;
    w.tmem_slot = reinterpret_cast<uint32_t *>(x + 12);
    w.tok = reinterpret_cast<int *>(smem + k.o_tok);
    w.flag = w.tok + 256;
    return w;
}


// The same unit walk on every role: unit, rank, column range and stage count;
// false when the unit has no work for the tensor-core roles.
template <int MODE>
__device__ __forceinline__ bool ws_unit(const TmaKernelParams &k, const unsigned char *smem, int nruns, int64_t u,
                                        bool report, Unit &U, int &r, int &n0, int &n1, int &nt) {
    const LoraParams &p = k.p;
    U = decode_unit<128>(k, smem, nruns, u);
    r = unit_rank(p, U, report);
    n0 = n1 = 0;
    nt = 0;
    if (MODE != kModeShrink) {
        column_range(p, U.nb, 0, 1, &n0, &n1);
        nt = n1 > n0 ? (n1 - n0 + kWsCols - 1) / kWsCols : 0;
    }
    return r > 0 && (MODE == kModeShrink || nt > 0);
}

// ------------------------------------------------------------------------------------- producer
template <int MODE, int STREAM>
__device__ void ws_producer(const TmaKernelParams &k, unsigned char *smem, int nruns, int64_t nunits) {
    // the first stream of the mode loads each tile's token list
    constexpr bool kLoadsTok = (STREAM == 0) == (MODE != kModeExpand);
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const WsBars W = ws_bars(k, smem);
    const int cR = p.c * p.R;
    const int nkc = (int)((p.K + 63) / 64);
    uint32_t sh_i = 0, ex_i = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit U;
        int r, n0, n1, nt;
        if (!ws_unit<MODE>(k, smem, nruns, u, kLoadsTok && lane == 0, U, r, n0, n1, nt)) continue;
        const int tb = uc & 1;
        int *tok = W.tok + tb * 128;
        if (kLoadsTok) {
            mbar_wait(&W.tok_empty[tb], ((uc >> 1) & 1) ^ 1, p.status, kStatusTimeout);
            for (int m = lane; m < 128; m += 32) {
                int t = -1;
                if (m < U.M) {
                    t = p.permutation[U.p0 + m];
                    if (t < 0 || t >= p.num_tokens) {
                        atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
                        t = -1;
                    }
                }
                tok[m] = t;
            }
            __syncwarp();
            const int tf = tok[0];
            bool mine = true;
            for (int m = lane; m < U.M; m += 32) mine = mine && tok[m] == tf + m;
            const bool cg = __all_sync(0xffffffffu, mine) && tf >= 0 && k.row_tma;
            if (lane == 0) W.flag[tb] = cg ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&W.tok_full[tb]);
        } else {
            mbar_wait(&W.tok_full[tb], (uc >> 1) & 1, p.status, kStatusTimeout);
        }
        const int t0 = tok[0];
        const bool contig = W.flag[tb] != 0;
        const int tfill = t0 >= 0 ? t0 : 0;
        auto grow = [&](int m) { return m < U.M && tok[m] >= 0 ? tok[m] : tfill; };
        ++uc;

        if (STREAM == 0 && MODE != kModeExpand) {
            for (int ci = 0; ci < nkc; ++ci) {
                const int s = sh_i % k.S1;
                mbar_wait(&W.sh_empty[s], ((sh_i / k.S1) & 1) ^ 1, p.status, kStatusTimeout);
                unsigned char *xs = smem + k.o_sh + s * k.sh_stage;
                const int k0 = ci * 64;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&W.sh_full[s], k.a_rows * 128 + 128 * 128);
                    tma_load_2d(xs + k.sh_a, &k.tmA, k0, U.w * cR, &W.sh_full[s]);
                    if (contig) tma_load_2d(xs, &k.tmX, k0, t0, &W.sh_full[s]);
                }
                if (!contig) {
                    // lane l: rows 4l .. 4l+3 in one TMA gather; rows past the tile
                    // (and rows of an invalid token) read a valid row, never used
                    __syncwarp();  // after the byte count is posted
                    const int m = 4 * lane;
                    tma_gather4(xs + m * 128, &k.tmXg, k0, grow(m), grow(m + 1), grow(m + 2), grow(m + 3),
                                &W.sh_full[s]);
                }
                cp_async_mbar_arrive(&W.sh_full[s]);
                ++sh_i;
            }
        }
        if (STREAM == 1 && MODE != kModeShrink) {
            // Stages come in pairs (one MMA / epilogue step each); a unit with an
            // odd stage count ends with an empty stage.  The B tile lands on
            // b_full; two stages later this warp checks it landed, zeroes the
            // adapter padding columns [r, round16(r)) if the rank is ragged, and
            // only then adds the last arrival that makes the stage full.
            const bool base_tma = contig && p.accumulate;
            const int RK = (r + 15) & ~15;
            const int nst = (nt + 1) & ~1;
            const uint32_t g0 = ex_i;
            const int Bbytes = kWsCols * p.R * 2;
            const int pcB = p.R / 8, shB = pc_shift_of(pcB);
            // a stage is made full `lag` stages after it is issued: the ring must
            // still have room for those (the consumers release pairs)
            const int lag = min(2, k.S2 - 2);
            auto b_ready = [&](int i) {
                const uint32_t g = g0 + i;
                const int e = g % k.S2;
                mbar_wait(&W.b_full[e], (g / k.S2) & 1, p.status, kStatusTimeout);
                if (RK != r && i < nt) {
                    unsigned char *bs = smem + k.o_bring + e * Bbytes;
                    const int c0 = r >> 3, nc = (RK >> 3) - c0;
                    for (int idx = lane; idx < kWsCols * nc; idx += 32) {
                        const int n = idx / nc, ch = c0 + idx % nc;
                        uint16_t *q16 = reinterpret_cast<uint16_t *>(bs) + swz(n, ch, pcB, shB);
#pragma unroll
                        for (int e2 = 0; e2 < 8; ++e2)
                            if (ch * 8 + e2 >= r) q16[e2] = 0;
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&W.ex_full[e]);
            };
            for (int i = 0; i < nst; ++i) {
                const int e = ex_i % k.S2;
                mbar_wait(&W.ex_empty[e], ((ex_i / k.S2) & 1) ^ 1, p.status, kStatusTimeout);
                unsigned char *ys = smem + k.o_ex + e * kWsBaseBytes;
                const bool real = i < nt;
                const int x0 = n0 + i * kWsCols, x1 = min(n1, x0 + kWsCols);
                if (lane == 0) {
                    if (real) {
                        mbar_arrive_expect_tx(&W.b_full[e], Bbytes);
                        tma_load_2d(smem + k.o_bring + e * Bbytes, &k.tmB, 0, U.w * (int)p.N + x0, &W.b_full[e]);
                        mbar_arrive_expect_tx(&W.ex_full[e], base_tma ? kWsBaseBytes : 0);
                        if (base_tma) tma_load_2d(ys, &k.tmY, x0, t0, &W.ex_full[e]);
                    } else {
                        mbar_arrive(&W.b_full[e]);
                        mbar_arrive(&W.ex_full[e]);
                    }
                }
                if (real && p.accumulate && !base_tma) {
                    for (int idx = lane; idx < U.M * 8; idx += 32) {
                        const int m = idx >> 3, c8 = idx & 7;
                        const int col = x0 + 8 * c8;
                        const int t = tok[m];
                        if (t >= 0 && col < x1)
                            cp_async16(ys + m * 128 + ((c8 ^ (m & 7)) << 4), p.y + (int64_t)t * p.N + col, 16);
                    }
                }
                cp_async_mbar_arrive(&W.ex_full[e]);
                ++ex_i;
                if (i >= lag) b_ready(i - lag);
            }
            for (int i = max(0, nst - lag); i < nst; ++i) b_ready(i);
            __syncwarp();
            if (!kLoadsTok && lane == 0) mbar_arrive(&W.tok_empty[tb]);  // done with the token list
        }
    }
}

// ------------------------------------------------------------------------------------- MMA issuer
template <int MODE, int STREAM>
__device__ void ws_mma(const TmaKernelParams &k, unsigned char *smem, int nruns, int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const WsBars W = ws_bars(k, smem);
    const int nkc = (int)((p.K + 63) / 64);
    const int Rb = p.R * 2;
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    unsigned char *ah = smem + k.o_ah;
    uint32_t sh_i = 0, ex_i = 0, acc_i = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit U;
        int r, n0, n1, nt;
        if (!ws_unit<MODE>(k, smem, nruns, u, false, U, r, n0, n1, nt)) continue;
        const int cr = p.c * r;
        const int Nh = (cr + 15) & ~15;
        const int RK = (r + 15) & ~15;
        const int ksteps = RK / 16;
        if (STREAM == 0 && MODE != kModeExpand) {
            mbar_wait(W.hacc_empty, (uc & 1) ^ 1, p.status, kStatusTimeout);
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(128, Nh);
            for (int ci = 0; ci < nkc; ++ci) {
                const int s = sh_i % k.S1;
                mbar_wait(&W.sh_full[s], (sh_i / k.S1) & 1, p.status, kStatusTimeout);
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t xa = smem_u32(smem + k.o_sh + s * k.sh_stage);
                    const uint32_t aa = xa + (uint32_t)k.sh_a;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc_mma_bf16(tmem, smem_desc_kmajor(xa + ks * 32, 128), smem_desc_kmajor(aa + ks * 32, 128),
                                    idesc, ci > 0 || ks > 0);
                    tc_commit(&W.sh_empty[s]);
                }
                __syncwarp();
                ++sh_i;
            }
            if (lane == 0) tc_commit(W.hacc_full);
            __syncwarp();
        }
        if (STREAM == 1 && MODE != kModeShrink) {
            mbar_wait(W.ah_full, uc & 1, p.status, kStatusTimeout);
            tc_fence_after();
            // operand descriptor of h: tile 2j (hi) and 2j+1 (lo) are consecutive
            // 16 KB tiles, so their start addresses step by kTcAhBytes / 16
            const uint64_t dh0 = smem_desc_kmajor(smem_u32(ah), 128);
            constexpr uint64_t kTileStep = kTcAhBytes >> 4;
            const int Bbytes = kWsCols * Rb;
            const int npair = (nt + 1) / 2;
            for (int g = 0; g < npair; ++g) {
                const int ea = ex_i % k.S2, eb = (ex_i + 1) % k.S2;
                mbar_wait(&W.ex_full[ea], (ex_i / k.S2) & 1, p.status, kStatusTimeout);
                mbar_wait(&W.ex_full[eb], ((ex_i + 1) / k.S2) & 1, p.status, kStatusTimeout);
                const int a = acc_i & 1;
                mbar_wait(&W.acc_empty[a], ((acc_i >> 1) & 1) ^ 1, p.status, kStatusTimeout);
                tc_fence_after();
                if (lane == 0) {
                    const int x0 = n0 + g * kWsPairCols;
                    const int ncols = min(n1, x0 + kWsPairCols) - x0;  // a multiple of 16
                    // the pair's B tiles sit in consecutive slots: rows x0 .. x0 + 127
                    const uint64_t bdesc = smem_desc_kmajor(smem_u32(smem + k.o_bring + ea * Bbytes), Rb);
                    const uint32_t d0 = tmem + (uint32_t)(kWsAccCol + a * kWsPairCols);
                    int c0 = 0;
                    while (c0 < ncols) {
                        const int j = slice_at(p, x0 + c0);
                        const int c1 = j + 1 < p.c ? min(ncols, p.off[j + 1] - x0) : ncols;
                        const uint32_t idesc = idesc_bf16_f32(128, c1 - c0);
                        const uint64_t bd = bdesc + (uint64_t)((c0 * Rb) >> 4);
                        for (int ks = 0; ks < ksteps; ++ks) {
                            const uint64_t dhi = dh0 + (uint64_t)(2 * j) * kTileStep + 2 * ks;
                            tc_mma_bf16(d0 + c0, dhi, bd + 2 * ks, idesc, ks > 0);
                            tc_mma_bf16(d0 + c0, dhi + kTileStep, bd + 2 * ks, idesc, true);
                        }
                        c0 = c1;
                    }
                    tc_commit(&W.acc_full[a]);
                }
                __syncwarp();
                ex_i += 2;
                ++acc_i;
            }
            if (lane == 0) tc_commit(W.ah_empty);  // the operand tiles are free once these MMAs are done
            __syncwarp();
        }
        ++uc;
    }
    // the last completions arrive before the CTA (and its barriers) goes away
    if (STREAM == 0 && MODE != kModeExpand && sh_i > 0)
        mbar_wait(&W.sh_empty[(sh_i - 1) % k.S1], ((sh_i - 1) / k.S1) & 1, p.status, kStatusTimeout);
    if (STREAM == 1 && MODE != kModeShrink && uc > 0) mbar_wait(W.ah_empty, (uc - 1) & 1, p.status, kStatusTimeout);
}

// ------------------------------------------------------------------------------------- epilogue
__device__ __forceinline__ void ah_put(unsigned char *ah, int j, int m, int kk, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    const int off = m * 128 + (((kk >> 3) ^ (m & 7)) << 4) + (kk & 7) * 2;
    *reinterpret_cast<__nv_bfloat16 *>(ah + (2 * j) * kTcAhBytes + off) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(ah + (2 * j + 1) * kTcAhBytes + off) = lo;
}

template <int MODE>
__device__ void ws_epilogue(const TmaKernelParams &k, unsigned char *smem, int nruns, int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int quarter = warp & 3;          // TMEM lanes this warp may read
    const int half = (warp - 4) >> 2;      // 0 / 1: which 32-column half of a stage
    const int etid = threadIdx.x - 128;    // 0..255 among the epilogue threads
    const bool storer = etid == 0;
    const WsBars W = ws_bars(k, smem);
    unsigned char *ah = smem + k.o_ah;
    const int row = 32 * quarter + lane;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    uint32_t ex_i = 0, acc_i = 0, uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        Unit U;
        int r, n0, n1, nt;
        if (!ws_unit<MODE>(k, smem, nruns, u, false, U, r, n0, n1, nt)) {
            // Rank-0 slots: the shrink writes zero h rows, a non-accumulating
            // expand zero output rows.
            if (r == 0 && (MODE == kModeShrink || (MODE == kModeExpand && !p.accumulate))) {
                const int cR = p.c * p.R;
                for (int m = 0; m < U.M; ++m) {
                    const int t = p.permutation[U.p0 + m];
                    if (t < 0 || t >= p.num_tokens) continue;
                    if (MODE == kModeShrink) {
                        for (int col = etid; col < cR; col += 256) {
                            if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = 0.f;
                            else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(0.f);
                        }
                    } else {
                        for (int ch = etid; ch < (n1 - n0) / 8; ch += 256)
                            *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + n0 + 8 * ch) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            continue;
        }
        const int tb = uc & 1;
        mbar_wait(&W.tok_full[tb], (uc >> 1) & 1, p.status, kStatusTimeout);
        const int *tok = W.tok + tb * 128;
        const bool contig = W.flag[tb] != 0;
        const int cr = p.c * r;
        const int Nh = (cr + 15) & ~15;
        const int RK = (r + 15) & ~15;
        const int t_row = row < U.M ? tok[row] : -1;

        if (MODE != kModeExpand) {
            mbar_wait(W.hacc_full, uc & 1, p.status, kStatusTimeout);
            tc_fence_after();
            if (MODE == kModeFused) mbar_wait(W.ah_empty, (uc & 1) ^ 1, p.status, kStatusTimeout);
            for (int pc = half; pc * 32 < Nh; pc += 2) {
                __syncwarp();
                float v[32];
                tmem_ld32(tmem + lane_addr + (uint32_t)(pc * 32), v);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int hc = pc * 32 + e;
                    if (hc >= cr) break;
                    if (MODE == kModeShrink) {
                        if (t_row >= 0) {
                            if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t_row * p.ldh + hc] = v[e];
                            else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t_row * p.ldh + hc] = __float2bfloat16_rn(v[e]);
                        }
                    } else {
                        const int j = hc / r;
                        ah_put(ah, j, row, hc - j * r, row < U.M ? v[e] : 0.f);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(W.hacc_empty);
            if (MODE == kModeShrink) {  // columns [c*r, c*R) of h are zero
                if (t_row >= 0)
                    for (int col = cr + half; col < p.c * p.R; col += 2) {
                        if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t_row * p.ldh + col] = 0.f;
                        else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t_row * p.ldh + col] = __float2bfloat16_rn(0.f);
                    }
            } else if (half == 0) {  // operand columns [r, RK) of every slice are zero
                for (int j = 0; j < p.c; ++j)
                    for (int kk = r; kk < RK; ++kk) ah_put(ah, j, row, kk, 0.f);
            }
        } else {
            // expand-only: the operand tiles from h in global memory
            mbar_wait(W.ah_empty, (uc & 1) ^ 1, p.status, kStatusTimeout);
            for (int j = half; j < p.c; j += 2)
                for (int kk = 0; kk < RK; ++kk) {
                    float v = 0.f;
                    if (kk < r && t_row >= 0) {
                        const int64_t o = (int64_t)t_row * p.ldh + j * r + kk;
                        v = p.h_f32 ? reinterpret_cast<const float *>(p.h)[o]
                                    : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[o]);
                    }
                    ah_put(ah, j, row, kk, v);
                }
        }
        if (MODE != kModeShrink) {
            fence_proxy_async_smem();  // the operand tiles are read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(W.ah_full);

            const float sigma = p.scalings[U.w];
            const int npair = (nt + 1) / 2;
            for (int g = 0; g < npair; ++g) {
                const int ea = ex_i % k.S2, eb = (ex_i + 1) % k.S2;
                const int a = acc_i & 1;
                mbar_wait(&W.acc_full[a], (acc_i >> 1) & 1, p.status, kStatusTimeout);
                mbar_wait(&W.ex_full[ea], (ex_i / k.S2) & 1, p.status, kStatusTimeout);
                mbar_wait(&W.ex_full[eb], ((ex_i + 1) / k.S2) & 1, p.status, kStatusTimeout);
                // this warp: rows 32*quarter.., the pair's stage `half` (64 columns)
                const int st = 2 * g + half;
                const bool real = st < nt;
                const int e = half ? eb : ea;
                const int x0 = n0 + st * kWsCols, x1 = min(n1, x0 + kWsCols);
                unsigned char *ys = smem + k.o_ex + e * kWsBaseBytes;
                tc_fence_after();
                __syncwarp();
                float v[2][32];
                if (real) {
                    const uint32_t ta = tmem + lane_addr + (uint32_t)(kWsAccCol + a * kWsPairCols + 64 * half);
                    tmem_ld32(ta, v[0]);
                    tmem_ld32(ta + 32, v[1]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&W.acc_empty[a]);
                if (real && row < U.M) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        if (x0 + 8 * c8 < x1) {
                            uint4 *ptr = reinterpret_cast<uint4 *>(ys + row * 128 + ((c8 ^ (row & 7)) << 4));
                            const float *vv = &v[c8 >> 2][8 * (c8 & 3)];
                            uint4 bv = p.accumulate ? *ptr : make_uint4(0, 0, 0, 0);
                            float2 f;
                            f = unpack_bf16x2(bv.x); bv.x = pack_bf16x2(f.x + sigma * vv[0], f.y + sigma * vv[1]);
                            f = unpack_bf16x2(bv.y); bv.y = pack_bf16x2(f.x + sigma * vv[2], f.y + sigma * vv[3]);
                            f = unpack_bf16x2(bv.z); bv.z = pack_bf16x2(f.x + sigma * vv[4], f.y + sigma * vv[5]);
                            f = unpack_bf16x2(bv.w); bv.w = pack_bf16x2(f.x + sigma * vv[6], f.y + sigma * vv[7]);
                            *ptr = bv;
                        }
                    }
                }
                // A whole stage of consecutive tokens and 64 columns goes back as
                // one TMA box; anything else as 16-byte row pieces.
                const bool store_tma = real && contig && U.M == 128 && x1 - x0 == kWsCols;
                if (real && !store_tma) {
                    __syncwarp();
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int idx = lane + 32 * it, rr = idx >> 3, c8 = idx & 7;
                        const int row2 = 32 * quarter + rr, col = x0 + 8 * c8;
                        if (row2 < U.M && col < x1) {
                            const int t = tok[row2];
                            if (t >= 0)
                                *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) =
                                    *reinterpret_cast<const uint4 *>(ys + row2 * 128 + ((c8 ^ (row2 & 7)) << 4));
                        }
                    }
                }
                fence_proxy_async_smem();  // in-place writes before the TMA store / the next TMA fill
                named_bar_sync(kWsEpiBar, kWsEpiWarps * 32);
                if (storer) {
                    // the pair's slots are handed back once its stores have read them
                    bool any = false;
                    for (int hs = 0; hs < 2; ++hs) {
                        const int sst = 2 * g + hs;
                        if (sst >= nt) continue;
                        const int sx0 = n0 + sst * kWsCols;
                        if (contig && U.M == 128 && min(n1, sx0 + kWsCols) - sx0 == kWsCols) {
                            tma_store_2d(&k.tmY, sx0, tok[0], smem + k.o_ex + (hs ? eb : ea) * kWsBaseBytes);
                            any = true;
                        }
                    }
                    if (any) {
                        bulk_commit();
                        bulk_wait_read<0>();
                    }
                    mbar_arrive(&W.ex_empty[ea]);
                    mbar_arrive(&W.ex_empty[eb]);
                }
                ex_i += 2;
                ++acc_i;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.tok_empty[tb]);
        ++uc;
    }
    if (storer) bulk_wait<0>();
}

template <int RMAX, int MODE>
__global__ void __launch_bounds__(kWsThreads, 1) lora_ws_kernel(const __grid_constant__ TmaKernelParams k) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    // The carve-up assumes the dynamic window starts on a 1024-byte boundary
    // (no slack is reserved); refuse to run otherwise.
    if (smem != smem_raw) {
        griddep_wait();
        if (threadIdx.x == 0) atomicOr(k.p.status, kStatusTimeout);
        return;
    }
    const WsBars W = ws_bars(k, smem);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < k.S1; ++i) { mbar_init(&W.sh_full[i], 1 + 32); mbar_init(&W.sh_empty[i], 1); }
        for (int i = 0; i < k.S2; ++i) {
            mbar_init(&W.ex_full[i], 2 + 32);  // base bytes, every lane's row copies, B landed (and cleaned)
            mbar_init(&W.ex_empty[i], 1);
            mbar_init(&W.b_full[i], 1);
        }
        mbar_init(W.hacc_full, 1);
        mbar_init(W.hacc_empty, kWsEpiWarps);
        mbar_init(W.ah_full, kWsEpiWarps);
        mbar_init(W.ah_empty, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&W.acc_full[i], 1);
            mbar_init(&W.acc_empty[i], kWsEpiWarps);
            mbar_init(&W.tok_full[i], 1);
            // released by the epilogue warps, and in the fused mode also by the expand producer
            mbar_init(&W.tok_empty[i], kWsEpiWarps + (MODE == kModeFused ? 1 : 0));
        }
        fence_mbar_init();
        prefetch_tmap(&k.tmA);
        prefetch_tmap(&k.tmB);
        prefetch_tmap(&k.tmX);
        prefetch_tmap(&k.tmY);
        prefetch_tmap(&k.tmXg);
    }
    if (warp == 3) {  // one warp owns the TMEM accumulators of the CTA
        tmem_alloc(W.tmem_slot, kWsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    int nruns = 0;
    const int ntiles = build_run_table<128>(k, smem, &nruns);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = *W.tmem_slot;
    const int64_t nunits = (int64_t)ntiles * k.p.nsplit;
    if (warp == 0) {
        if (MODE != kModeExpand) ws_producer<MODE, 0>(k, smem, nruns, nunits);
    } else if (warp == 1) {
        if (MODE != kModeShrink) ws_producer<MODE, 1>(k, smem, nruns, nunits);
    } else if (warp == 2) {
        if (MODE != kModeExpand) ws_mma<MODE, 0>(k, smem, nruns, nunits, tmem);
    } else if (warp == 3) {
        if (MODE != kModeShrink) ws_mma<MODE, 1>(k, smem, nruns, nunits, tmem);
    } else {
        ws_epilogue<MODE>(k, smem, nruns, nunits, tmem);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 3) {
        tc_fence_after();
        tmem_dealloc(tmem, kWsTmemCols);
    }
}

}  // namespace csgmv
