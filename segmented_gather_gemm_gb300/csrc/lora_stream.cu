// The streaming tcgen05 expand kernel for 128-token tiles (see lora_stream.cuh).
#include "lora_stream.cuh"

namespace csgmv {

constexpr int kOpLoCol = kStOpCols / 2;  // the lo half of an operand buffer
// stage pairs (st_mma): an even stage's B slot and accumulator have their
// neighbours next to them, and two stages fit one MMA of N = 128
static_assert(kStBSlots % 2 == 0 && kStAcc % 2 == 0 && kStCols == 64, "stage pairs");
constexpr int kStOpBar = 1;              // named barrier of the operand warps

struct StBars {
    uint64_t *b_full, *b_empty;      // [Sb]
    uint64_t *b_ready;               // [Sb] B tile landed and its padding columns zeroed
    int *bpad;                       // [Sb] rank r | round16(r) << 16 of the tile in each B slot
    uint64_t *y_full, *y_empty;      // [Sy]
    uint64_t *acc_full, *acc_empty;  // [kStAcc]
    uint64_t *op_full, *op_empty;    // [2]
    uint32_t *tmem_slot;
    int *tok;   // [2][128] token of each tile row (-1: none)
    int *flag;  // [2] the tile's rows are consecutive tokens; [2, 6) scratch
};

__device__ __forceinline__ StBars st_bars(const StreamParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    StBars w;
    w.b_full = b;
    w.b_empty = b + k.Sb;
    w.y_full = b + 2 * k.Sb;
    w.y_empty = w.y_full + k.Sy;
    w.acc_full = w.y_empty + k.Sy;
    w.acc_empty = w.acc_full + kStAcc;
    w.op_full = w.acc_empty + kStAcc;
    w.op_empty = w.op_full + 2;
    w.b_ready = w.op_empty + 2;
    w.tmem_slot = reinterpret_cast<uint32_t *>(w.b_ready + k.Sb);
    w.bpad = reinterpret_cast<int *>(w.tmem_slot + 4);
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

// ------------------------------------------------------------------------------------- producers
// B tiles: they need no token list, so this warp runs ahead of the operand
// tiles by as many stages as the B ring holds.  A tile of a slot whose rank r
// is not a multiple of 16 carries adapter padding in columns [r, round16(r))
// (even NaN), which must be zero before its MMAs: this warp zeroes it D
// stages after issuing the tile (waiting for it to land), then releases the
// slot to the MMA warp (b_ready), so the padding pass is off the MMA warp's
// per-stage chain.  D < Sb: the slot the producer waits to refill was
// released D stages of issue earlier.
__device__ void st_b_producer(const StreamParams &k, unsigned char *smem, const int *tables, int nruns,
                              int64_t nunits) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const StBars W = st_bars(k, smem);
    const uint32_t Bbytes = (uint32_t)kStCols * p.R * 2;  // kStBoxes boxes of 64 B rows
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    const uint32_t D = (uint32_t)max(1, k.Sb / 2);
    auto release = [&](uint32_t gz) {
        const int sb = gz % k.Sb;
        mbar_wait(&W.b_full[sb], (gz / k.Sb) & 1, p.status, kStatusTimeout);
        const int info = W.bpad[sb];
        const int r = info & 0xffff, RK = info >> 16;
        if (RK != r) {
            // lane l takes rows l and l + 32: whole padding chunks as one
            // 16-byte store, a chunk holding column r element by element
            unsigned char *bs = smem + k.o_bring + sb * k.b_slot_bytes;
            const int cpart = r >> 3, nc = (RK >> 3) - cpart;
#pragma unroll
            for (int h2 = 0; h2 < kStCols / 32; ++h2) {
                const int n = lane + 32 * h2;
                for (int ch = cpart; ch < cpart + nc; ++ch) {
                    uint16_t *q16 = reinterpret_cast<uint16_t *>(bs) + swz(n, ch, pcB, shB);
                    if (ch * 8 >= r) {
                        *reinterpret_cast<uint4 *>(q16) = make_uint4(0u, 0u, 0u, 0u);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (ch * 8 + e >= r) q16[e] = 0;
                    }
                }
            }
            fence_proxy_async_smem();  // the tensor core reads these columns
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.b_ready[sb]);
    };
    uint32_t g = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, false, U, r)) continue;
        // row in the 2-D view of B_j of column x of the unit's slice
        const int brow = U.w * p.b_rows[U.j] + p.b_row0[U.j] - p.off[U.j];
        for (int i = 0; i < U.nt; ++i, ++g) {
            const int sb = g % k.Sb;
            const int x0 = U.n0 + i * kStCols;
            mbar_wait(&W.b_empty[sb], ((g / k.Sb) & 1) ^ 1, p.status, kStatusTimeout);
            if (lane == 0) {
                unsigned char *bs = smem + k.o_bring + sb * k.b_slot_bytes;
                W.bpad[sb] = r | (((r + 15) & ~15) << 16);
                mbar_arrive_expect_tx(&W.b_full[sb], Bbytes);
#pragma unroll
                for (int bx = 0; bx < kStBoxes; ++bx)
                    tma_load_2d(bs + bx * 64 * p.R * 2, &k.tmB[U.j], 0, brow + x0 + 64 * bx, &W.b_full[sb]);
            }
            __syncwarp();
            if (g >= D) release(g - D);
        }
    }
    for (uint32_t gz = g > D ? g - D : 0; gz < g; ++gz) release(gz);
}

// Base rows of every stage, through the tile's token list.
__device__ void st_producer(const StreamParams &k, unsigned char *smem, const int *tables, int nruns,
                            int64_t nunits) {
    const LoraParams &p = k.p;
    const int lane = threadIdx.x & 31;
    const StBars W = st_bars(k, smem);
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
        for (int i = 0; i < U.nt; ++i, ++g) {
            const int sy = g % k.Sy;
            const int x0 = U.n0 + i * kStCols;
            mbar_wait(&W.y_empty[sy], ((g / k.Sy) & 1) ^ 1, p.status, kStatusTimeout);
            unsigned char *ys = smem + k.o_yring + sy * k.y_slot_bytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&W.y_full[sy],
                                      !p.accumulate ? 0 : contig ? kStBoxes * row_box_bytes(U.M) : kStBoxes * kStTileBytes);
                if (p.accumulate && contig)
#pragma unroll
                    for (int bx = 0; bx < kStBoxes; ++bx)
                        load_row_boxes(ys + bx * kStTileBytes, k.tmY, x0 + 64 * bx, t0, U.M, &W.y_full[sy]);
            }
            if (p.accumulate && !contig) {
                // lane l: tile rows 4l .. 4l+3 in one gather per box; rows past the
                // tile (or of an invalid token) read a valid row that is never used
                __syncwarp();  // after the byte count is posted
                const int m = 4 * lane;
                auto grow = [&](int mm) {
                    const int t = mm < U.M ? tok[mm] : -1;
                    return t >= 0 ? t : tfill;
                };
                const int r0 = grow(m), r1 = grow(m + 1), r2 = grow(m + 2), r3 = grow(m + 3);
#pragma unroll
                for (int bx = 0; bx < kStBoxes; ++bx)
                    tma_gather4(ys + bx * kStTileBytes + m * 128, &k.tmYg, x0 + 64 * bx, r0, r1, r2, r3,
                                &W.y_full[sy]);
            }
            __syncwarp();
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
        const uint32_t ahi = tmem + (uint32_t)(kStOpCol0 + b * kStOpCols), alo = ahi + kOpLoCol;
        // Stages go to the tensor core in pairs where they can: stage g (even)
        // and g + 1 sit in neighbouring B slots and TMEM accumulators, so one
        // MMA of N = 128 does both (half the MMA instructions, whose issue
        // sets this warp's pace).
        for (int i = 0; i < U.nt;) {
            const int n = (g & 1) == 0 && i + 1 < U.nt ? 2 : 1;
            const int sb = g % k.Sb;
            const int a = g % kStAcc;
            // landed, padding columns [r, RK) zeroed by the B producer
            for (int j = 0; j < n; ++j)
                mbar_wait(&W.b_ready[(g + j) % k.Sb], ((g + j) / k.Sb) & 1, p.status, kStatusTimeout);
            for (int j = 0; j < n; ++j)
                mbar_wait(&W.acc_empty[(g + j) % kStAcc], (((g + j) / kStAcc) & 1) ^ 1, p.status, kStatusTimeout);
            tc_fence_after();
            if (lane == 0) {
                const int x0 = U.n0 + i * kStCols;
                const int ncols = min(U.n1, x0 + n * kStCols) - x0;
                const uint32_t idesc = idesc_bf16_f32(128, (ncols + 15) & ~15);
                const uint32_t bsa = smem_u32(smem + k.o_bring + sb * k.b_slot_bytes);
                const uint32_t d = tmem + (uint32_t)(a * kStCols);
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint64_t bd = smem_desc_kmajor(bsa + ks * 32, Rb);
                    tc_mma_bf16_tmem_a(d, ahi + ks * 8, bd, idesc, ks > 0);
                    tc_mma_bf16_tmem_a(d, alo + ks * 8, bd, idesc, true);
                }
                for (int j = 0; j < n; ++j) tc_commit(&W.b_empty[(g + j) % k.Sb]);
                for (int j = 0; j < n; ++j) tc_commit(&W.acc_full[(g + j) % kStAcc]);
            }
            __syncwarp();
            i += n;
            g += n;
        }
        ++uc;
    }
    // the last slot releases land before the CTA (and its barriers) goes away
    for (uint32_t gg = g > (uint32_t)k.Sb ? g - k.Sb : 0; gg < g; ++gg)
        mbar_wait(&W.b_empty[gg % k.Sb], (gg / k.Sb) & 1, p.status, kStatusTimeout);
}

// ------------------------------------------------------------------------------------- operands
// h[t][col .. col+7] as fp32 (0 past `r` columns of the slice, i.e. col >= lim).
// fp32 h held as partial sums over parts of K is summed part by part, in order.
__device__ __forceinline__ void st_h8(const LoraParams &p, int parts, int t, int col, int lim, float (&v)[8]) {
    const int64_t o = (int64_t)t * p.ldh + col;
    if (p.h_f32) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        for (int part = 0; part < parts; ++part) {
            const float *h = reinterpret_cast<const float *>(p.h) + part * p.h_plane + o;
            if (col + 8 <= lim && ((o + part * p.h_plane) & 3) == 0) {
                const float4 a = *reinterpret_cast<const float4 *>(h), b = *reinterpret_cast<const float4 *>(h + 4);
                v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
                v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] += col + e < lim ? h[e] : 0.f;
            }
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
                            int64_t nunits, uint32_t tmem) {
    const LoraParams &p = k.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;  // TMEM lanes (tile rows) 32q .. 32q+31
    const int row = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const StBars W = st_bars(k, smem);
    // partial-sum planes of h: as the shrink chose them (at most h_parts)
    const int parts = p.h_parts_dev ? max(1, min(*p.h_parts_dev, p.h_parts)) : p.h_parts;
    uint32_t uc = 0;
    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        StUnit U;
        int r;
        if (!st_unit(k, tables, nruns, u, row == 0, U, r)) continue;
        const int b = uc & 1;
        mbar_wait(&W.op_empty[b], ((uc >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        int *tok = W.tok + b * 128;
        int t = -1;
        if (row < U.M) {
            t = p.permutation[U.p0 + row];
            if (t < 0 || t >= p.num_tokens) {
                atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION);
                t = -1;
            }
        }
        tok[row] = t;
        named_bar_sync(kStOpBar, 128);
        const int t0 = tok[0];
        const bool wall = __all_sync(0xffffffffu, row >= U.M || t == t0 + row);
        if (lane == 0) W.flag[2 + q] = wall ? 1 : 0;
        named_bar_sync(kStOpBar, 128);
        if (row == 0) W.flag[b] = (W.flag[2] && W.flag[3] && W.flag[4] && W.flag[5] && t0 >= 0) ? 1 : 0;

        // this row of h (columns [0, RK) of slice j) as bf16 hi / lo pairs
        const int RK = (r + 15) & ~15;
        const int col0 = U.j * r;
        const uint32_t ob = tmem + lane_base + (uint32_t)(kStOpCol0 + b * kStOpCols);
        for (int kb = 0; kb < RK / 16; ++kb) {
            float v[16];
            if (t >= 0) {
                float (&v0)[8] = *reinterpret_cast<float (*)[8]>(&v[0]);
                float (&v1)[8] = *reinterpret_cast<float (*)[8]>(&v[8]);
                st_h8(p, parts, t, col0 + kb * 16, col0 + r, v0);
                st_h8(p, parts, t, col0 + kb * 16 + 8, col0 + r, v1);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = 0.f;
            }
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) split_pair(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
            tmem_st8(ob + (uint32_t)(kb * 8), hi);
            tmem_st8(ob + (uint32_t)(kOpLoCol + kb * 8), lo);
        }
        tmem_wait_st();
        tc_fence_before();  // the operand columns are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&W.op_full[b]);
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
            if ((int)(g % kStTeams) != team) continue;
            const int sy = g % k.Sy;
            const int a = g % kStAcc;
            mbar_wait(&W.acc_full[a], (g / kStAcc) & 1, p.status, kStatusTimeout);
            mbar_wait(&W.y_full[sy], (g / k.Sy) & 1, p.status, kStatusTimeout);
            tc_fence_after();
            const int x0 = U.n0 + i * kStCols;
            const int ncols = min(U.n1, x0 + kStCols) - x0;
            const bool full = box && ncols == kStCols;
            unsigned char *ys = smem + k.o_yring + sy * k.y_slot_bytes;
#pragma unroll
            for (int bx = 0; bx < kStBoxes; ++bx) {
                __syncwarp();  // tcgen05.ld is warp-wide
                float v[64];
                tmem_ld64(tmem + lane_base + (uint32_t)(a * kStCols + 64 * bx), v);
                if (bx == kStBoxes - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&W.acc_empty[a]);
                }
                unsigned char *yb = ys + bx * kStTileBytes;
                if (row < U.M && (full || trow >= 0)) {
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        if (64 * bx + 8 * c8 < ncols) {
                            uint4 *ptr = reinterpret_cast<uint4 *>(yb + row * 128 + ((c8 ^ (row & 7)) << 4));
                            const float *vv = &v[8 * c8];
                            uint4 bv = p.accumulate ? *ptr : make_uint4(0, 0, 0, 0);
                            float2 f;
                            f = unpack_bf16x2(bv.x); bv.x = pack_bf16x2(f.x + sigma * vv[0], f.y + sigma * vv[1]);
                            f = unpack_bf16x2(bv.y); bv.y = pack_bf16x2(f.x + sigma * vv[2], f.y + sigma * vv[3]);
                            f = unpack_bf16x2(bv.z); bv.z = pack_bf16x2(f.x + sigma * vv[4], f.y + sigma * vv[5]);
                            f = unpack_bf16x2(bv.w); bv.w = pack_bf16x2(f.x + sigma * vv[6], f.y + sigma * vv[7]);
                            if (full) *ptr = bv;
                            else *reinterpret_cast<uint4 *>(p.y + (int64_t)trow * p.N + x0 + 64 * bx + 8 * c8) = bv;
                        }
                    }
                }
            }
            fence_proxy_async_smem();  // in-place rows before the TMA store reads them; reads before a refill
            __syncwarp();
            if (lane == 0) {
                if (full) {  // the slot goes back once the stores have read this warp's rows
#pragma unroll
                    for (int bx = 0; bx < kStBoxes; ++bx)
                        tma_store_2d(&k.tmYs, x0 + 64 * bx, t0 + 32 * q, ys + bx * kStTileBytes + 32 * q * 128);
                    bulk_commit();
                    bulk_wait_read<0>();
                }
                mbar_arrive(&W.y_empty[sy]);
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
        for (int i = 0; i < k.Sb; ++i) {
            mbar_init(&W.b_full[i], 1);
            mbar_init(&W.b_empty[i], 1);
            mbar_init(&W.b_ready[i], 1);
        }
        for (int i = 0; i < k.Sy; ++i) {
            mbar_init(&W.y_full[i], 1);
            mbar_init(&W.y_empty[i], 4);  // the four warps of the team that takes the stage
        }
        for (int i = 0; i < kStAcc; ++i) {
            mbar_init(&W.acc_full[i], 1);
            mbar_init(&W.acc_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&W.op_full[i], 4);                 // the operand warps
            mbar_init(&W.op_empty[i], 1 + kStEpiWarps);  // producer + epilogue warps
        }
        fence_mbar_init();
        for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmB[j]);
        for (int l = 0; l < kRowBoxLevels; ++l) prefetch_tmap(&k.tmY[l]);
        prefetch_tmap(&k.tmYs);
        prefetch_tmap(&k.tmYg);
    }
    if (warp == 1) {  // one warp owns the TMEM accumulators of the CTA
        tmem_alloc(W.tmem_slot, kStTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    int nruns = 0;
    int *tables = reinterpret_cast<int *>(smem + k.o_run);
    const int ntiles = build_run_table_raw<128, true>(k.p, k.max_segments, k.runcap, tables, &nruns);  // ends with __syncthreads
    tc_fence_after();
    const uint32_t tmem = *W.tmem_slot;
    const int64_t nunits = (int64_t)ntiles * k.upt;
    if (warp == 0) st_producer(k, smem, tables, nruns, nunits);
    else if (warp == 1) st_mma(k, smem, tables, nruns, nunits, tmem);
    else if (warp == 2) st_b_producer(k, smem, tables, nruns, nunits);
    else if (warp >= kStOpWarp0 && warp < kStEpiWarp0) st_operands(k, smem, tables, nruns, nunits, tmem);
    else if (warp >= kStEpiWarp0) st_epilogue(k, smem, tables, nruns, nunits, tmem);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kStTmemCols);
    }
}

const void *lora_kernel_stream() { return reinterpret_cast<const void *>(lora_stream_expand_kernel); }

}  // namespace csgmv
