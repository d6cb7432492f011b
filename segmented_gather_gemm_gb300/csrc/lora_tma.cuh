// Shrink, expand and fused shrink->expand kernels of the csgmv LoRA path
// (sglang chunked_backend.py run_lora_a_sgemm, run_lora_b_sgemm, run_qkv_lora,
// run_gate_up_lora; shapes from base_backend.py), driven by the TMA engine.
//
// Work units.  The batch info orders tokens by slot and cuts each slot's run
// into chunk-sized segments.  Each CTA first rebuilds, in shared memory, the
// list of slot runs (maximal runs of consecutive segments on one slot) and
// cuts every run into tiles of at most TM tokens, so no unit is empty and
// consecutive same-slot segments share a tile whatever the chunk size.  A unit
// is (tile, column block); clusters walk the unit list with a fixed stride.
//
// Per unit a cluster of CS CTAs:
//   shrink  CTA q multiplies the tile's x rows by A[w] over its 1/CS share of
//           K: the permuted x rows arrive by coalesced 16-byte cp.async, the
//           A rows of each 64-wide K chunk by 2D TMA (128-byte swizzle); both
//           complete on the stage's mbarrier; mma.sync m16n8k16, fp32
//           accumulators;
//   reduce  partials go to shared memory, CTA q sums its 1/CS of the rows over
//           the cluster through distributed shared memory, and every consumer
//           warp then pulls the fp32 h it needs from the owning CTA straight
//           into registers as bf16 hi + lo fragment pairs;
//   expand  CTA q streams its share of the output columns: base rows by
//           cp.async, B[w] column tiles by 2D TMA, y = base + sigma h B^T on the
//           tensor cores, and y back with 16-byte stores.
// All sixteen warps gather rows, do the math and store; when a stage is free
// (its mbarrier says every warp is done with it) thread 0 also issues the
// stage's single weight-tile TMA box.  A stage is full when the TMA bytes and
// every thread's cp.async have landed (cp.async.mbarrier.arrive), so no
// block-wide barrier sits in the streaming loops; all waits are bounded.
// Rows go through the load/store units rather than TMA gather: a TMA
// instruction costs its issuing thread tens to a hundred cycles, so 4-row
// gathers cannot keep HBM busy, while one warp-wide cp.async moves 512 B.
// h never leaves the chip in the fused mode; the shrink-only mode writes it to
// global memory after the reduction and the expand-only mode (cluster of one)
// reads it from there.
#pragma once

#include <cuda.h>

#include "csgmv_internal.h"
#include "device_utils.cuh"

namespace csgmv {

constexpr int kConsumerWarps = 16;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kTmaThreads = kConsumerThreads;  // every warp gathers, computes and stores
constexpr int kBarConsumers = 1;               // named barrier id
constexpr int kStatusTimeout = 64;                   // device status bit: a bounded wait ran out

struct TmaKernelParams {
    CUtensorMap tmA;    // A (L*c*R rows, K): box 64 x round16(c*R), 128B swizzle
    CUtensorMap tmB;    // B (L*N rows, R):   box R x NT, swizzle of the R*2-byte row
    CUtensorMap tmX;    // x (s rows, K): box 64 x TM, 128B swizzle (128-token tiles)
    CUtensorMap tmY;    // base / y (s rows, N): box 64 x TM, 128B swizzle (128-token tiles)
    CUtensorMap tmXg;   // x, box 64 x 1, 128B swizzle, for 4-row gathers
    CUtensorMap tmBs[kMaxSlices];  // B as separate slice tensors (p.b_tuple): box R x 64 of slice j
    int row_tma;        // 1: tmX / tmY are valid; tiles of consecutive tokens load rows by TMA
    LoraParams p;
    int S1, S2;        // shrink / expand ring depth
    int runcap;        // slot-run capacity of the run table
    int max_segments;
    int o_bar, o_run, o_tok, o_sh, o_hpart, o_hred, o_ex;
    int sh_stage, sh_a;  // shrink stage bytes, A offset inside a stage
    int a_rows;          // rows of the A box (round16(c*R))
    int ex_stage, ex_b;  // expand stage bytes, B offset inside a stage
    int hp;            // floats per hpart / hred row
    int o_tc;          // tensor-core expand: acc_full[2], acc_empty[2], TMEM base address
    int o_ah;          // tensor-core expand: h of every slice as bf16 hi / lo operand tiles
    int ah_slices;     // tensor-core expand: slices one CTA's column range can span (operand tile pairs)
    int o_bring;       // warp-specialized kernel: B tiles of the expand stages (consecutive slots)
    int xpitch, ypitch;  // small-tile kernel: bytes per staged x row / base row
    int kc_per;          // small-tile kernel: 64-wide K chunks staged per CTA
    int wscr_off;        // small-tile kernel: per-warp epilogue scratch, bytes after o_hpart
};

// Tensor-core (tcgen05) expand: 128-token tile x 128-column stage, the fp32
// accumulator of a stage in TMEM (two stages in flight, 256 columns).
constexpr int kTcCols = 128;
constexpr int kTcTmemCols = 2 * kTcCols;
constexpr int kTcAhBytes = 128 * 128;  // one 128 x 64 bf16 operand tile (128-byte rows)

template <int TM, bool TC = false>
struct Geo {
    static constexpr int WM = TM / 16;                    // consumer warps along tokens
    static constexpr int WN = kConsumerWarps / WM;        // consumer warps along columns
    static constexpr int NB64 = TC ? kTcCols / 64 : (TM >= 128 ? 1 : (TM >= 64 ? 2 : 4));  // 64-column boxes per expand stage
    static constexpr int NT = 64 * NB64;                  // expand stage width
    static constexpr int WCOLS = NT / WN;                 // columns per consumer warp
    static constexpr int EXT = WCOLS / 8;                 // n8 tiles per consumer warp
};

struct Unit {
    int w, p0, M, nb;
};

struct Bars {
    uint64_t *sh_full, *sh_empty, *ex_full, *ex_empty;
};

__device__ __forceinline__ Bars bars_of(const TmaKernelParams &k, unsigned char *smem) {
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + k.o_bar);
    Bars r;
    r.sh_full = b;
    r.sh_empty = b + k.S1;
    r.ex_full = b + 2 * k.S1;
    r.ex_empty = b + 2 * k.S1 + k.S2;
    return r;
}

// Exclusive scan over the whole block; every thread must call it.
__device__ __forceinline__ int block_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < nw) scratch[lane] = w;
    }
    __syncthreads();
    int pre = (warp > 0 ? scratch[warp - 1] : 0) + inc - v;
    *total = scratch[nw - 1];
    __syncthreads();
    return pre;
}

// Cuts the slot runs (starts run_p0, ends run_end, slots run_w; adjacent and
// in position order) where the permutation is not consecutive; the cut runs
// replace them in the same arrays.  Within a slot run the stable sort keeps
// tokens in increasing order, so g(p) = permutation[p] - p never decreases
// there: a stretch of one run holds a gap exactly when g differs at its two
// ends, and each gap is found by a binary search.  Each thread takes one
// stretch of about s / threads positions; a stretch with more than kMaxGaps
// cuts is scanned position by position instead.  A gap this misses (an
// out-of-range entry breaks the order) only costs speed: every tile's rows
// are checked for consecutiveness before they are loaded as a box.
// `scratch` is followed by 3 * runcap ints of room.  Returns the new run
// count (0 and a status bit on overflow).  Every thread of the block calls it.
static __device__ __noinline__ int split_runs_at_gaps(const LoraParams &p, int runcap, int *run_p0, int *run_end,
                                                      int *run_w, int *scratch, int nruns) {
    constexpr int kMaxGaps = 8;
    int *sub_p0 = scratch + 32, *sub_w = sub_p0 + runcap, *sub_end = sub_w + runcap;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int first = nruns > 0 ? run_p0[0] : 0, last = nruns > 0 ? run_end[nruns - 1] : 0;
    const int stretch = max(1, (last - first + nt - 1) / nt);
    const int a = min(last, first + tid * stretch), b = min(last, a + stretch);
    auto g = [&](int pp) { return p.permutation[pp] - pp; };
    int r0 = 0;  // the run holding position a
    {
        int lo = 0, hi = nruns;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (run_p0[mid] <= a) lo = mid; else hi = mid;
        }
        r0 = lo;
    }
    // cut at x (a <= x < last): a run starts there, or x - 1 (same run) is not its predecessor token
    auto cut_at = [&](int x, int r) { return x == run_p0[r] || p.permutation[x] != p.permutation[x - 1] + 1; };
    int cuts[kMaxGaps];
    int nc = 0;
    bool linear = false;
    for (int u = a, r = r0; u < b && !linear; ++r) {
        const int v = min(b, run_end[r]);  // piece [u, v) of run r
        if (cut_at(u, r)) {
            if (nc == kMaxGaps) { linear = true; break; }
            cuts[nc++] = u;
        }
        int lo = u;
        const int gv = g(v - 1);
        while (lo < v - 1 && g(lo) != gv) {
            const int gl = g(lo);
            int L = lo + 1, H = v - 1;  // first x in (lo, v) with g(x) > g(lo)
            while (L < H) {
                const int M = (L + H) >> 1;
                if (g(M) > gl) H = M; else L = M + 1;
            }
            if (nc == kMaxGaps) { linear = true; break; }
            cuts[nc++] = L;
            lo = L;
        }
        u = v;
    }
    int count = nc;
    if (linear) {
        count = 0;
        for (int x = a, r = r0; x < b; ++x) {
            while (r + 1 < nruns && run_p0[r + 1] <= x) ++r;
            count += cut_at(x, r);
        }
    }
    int tot;
    const int pre = block_scan(count, scratch, &tot);
    int idx = pre;
    auto put = [&](int x, int r) {
        if (idx < runcap) {
            sub_p0[idx] = x;
            sub_w[idx] = run_w[r];
            sub_end[idx] = run_end[r];
        }
        ++idx;
    };
    if (linear) {
        for (int x = a, r = r0; x < b; ++x) {
            while (r + 1 < nruns && run_p0[r + 1] <= x) ++r;
            if (cut_at(x, r)) put(x, r);
        }
    } else {
        int r = r0;
        for (int i = 0; i < nc; ++i) {
            while (r + 1 < nruns && run_p0[r + 1] <= cuts[i]) ++r;
            put(cuts[i], r);
        }
    }
    int nsub = tot;
    if (nsub > runcap) {
        if (tid == 0) atomicOr(p.status, CSGMV_STATUS_CAPACITY);
        nsub = 0;
    }
    __syncthreads();
    for (int i = tid; i < nsub; i += nt) {
        run_p0[i] = sub_p0[i];
        run_w[i] = sub_w[i];
        run_end[i] = i + 1 < nsub ? min(sub_p0[i + 1], sub_end[i]) : sub_end[i];
    }
    __syncthreads();
    return nsub;
}

// Slot runs of the batch info and their token tiles (see the file comment).
// Returns the number of tiles; the tables live in shared memory.
// `tables` holds 5 * runcap + 1 + 32 ints (8 * runcap + 1 + 32 with SPLIT);
// every thread of the block calls it.
//
// SPLIT: runs are also cut wherever the permutation is not consecutive
// (permutation[p] != permutation[p-1] + 1, i.e. between two requests on one
// slot), so every tile holds consecutive tokens and moves its rows as TMA
// boxes.  A request's tokens stay together in the stable sort, so this gives
// at most one run per request: the run capacity max_bs + max_loras holds.
template <int TM, bool SPLIT = false>
__device__ int build_run_table_raw(const LoraParams &p, int max_segments, int runcap, int *tables,
                                   int *nruns_out) {
    int *run_seg = tables;
    int *run_p0 = run_seg + runcap;
    int *run_len = run_p0 + runcap;
    int *run_w = run_len + runcap;
    int *run_tp = run_w + runcap;        // [runcap + 1]
    int *scratch = run_tp + runcap + 1;  // [32]
    const int tid = threadIdx.x, nt = blockDim.x;
    griddep_wait();  // the batch info may come from the kernel launched just before
    // Every word a thread needs is loaded in one round, bounded by the
    // capacity rather than by the segment count (which is loaded alongside).
    const int cap = max_segments;
    const int nseg_raw = *p.num_segments_dev;
    // each pass gives thread tid the G consecutive segments k0 + G*tid + j:
    // every load of a pass goes out before the first is used, and one block
    // scan numbers the runs of G * nt segments
    constexpr int G = 4;
    int carry = 0;
    for (int k0 = 0; k0 < cap; k0 += G * nt) {
        const int s0 = k0 + G * tid;
        int w[G + 2], ip[G + 1];  // w[j + 1] = weight_indices[s0 + j], j = -1 .. G; ip[j] = seg_indptr[s0 + j]
#pragma unroll
        for (int j = -1; j <= G; ++j) {
            const int s = s0 + j;
            w[j + 1] = s >= 0 && s < cap ? p.weight_indices[s] : -1;
        }
#pragma unroll
        for (int j = 0; j <= G; ++j) {
            const int s = s0 + j;
            ip[j] = s <= cap ? p.seg_indptr[s] : 0;
        }
        const int nseg = max(0, min(nseg_raw, cap));
        if (k0 >= nseg) break;
        int st[G], en[G], cnt = 0;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const int s = s0 + j;
            st[j] = s < nseg && (s == 0 || w[j + 1] != w[j]);
            en[j] = s < nseg && (s == nseg - 1 || w[j + 2] != w[j + 1]);
            cnt += st[j];
        }
        int tot;
        int run = carry + block_scan(cnt, scratch, &tot) - 1;  // run of the segment before s0
#pragma unroll
        for (int j = 0; j < G; ++j) {
            run += st[j];  // run of segment s0 + j
            if (st[j] && run < runcap) {
                run_w[run] = w[j + 1];
                run_p0[run] = max(0, min(ip[j], p.num_tokens));
            }
            if (en[j] && run >= 0 && run < runcap) run_len[run] = max(0, min(ip[j + 1], p.num_tokens));  // run end for now
        }
        carry += tot;
    }
    int nruns = carry;
    if (nruns > runcap) {
        if (tid == 0) atomicOr(p.status, CSGMV_STATUS_CAPACITY);
        nruns = 0;
    }
    __syncthreads();
    if constexpr (SPLIT) nruns = split_runs_at_gaps(p, runcap, run_p0, run_len, run_w, scratch, nruns);
    int tcarry = 0;
    for (int r0 = 0; r0 < nruns; r0 += nt) {
        const int r = r0 + tid;
        int tiles = 0;
        if (r < nruns) {
            const int len = max(0, run_len[r] - run_p0[r]);
            run_len[r] = len;
            tiles = (len + TM - 1) / TM;
        }
        int tot;
        const int pre = block_scan(tiles, scratch, &tot);
        if (r < nruns) run_tp[r] = tcarry + pre;
        tcarry += tot;
    }
    if (tid == 0) run_tp[nruns] = tcarry;
    __syncthreads();
    *nruns_out = nruns;
    return tcarry;
}

template <int TM>
__device__ int build_run_table(const TmaKernelParams &k, unsigned char *smem, int *nruns_out) {
    return build_run_table_raw<TM>(k.p, k.max_segments, k.runcap, reinterpret_cast<int *>(smem + k.o_run),
                                   nruns_out);
}

// Slot, first sorted position and size of token tile `tile` (run table of
// build_run_table_raw).
template <int TM>
__device__ __forceinline__ Unit tile_of(const int *tables, int runcap, int nruns, int tile) {
    const int *run_seg = tables;
    const int *run_p0 = run_seg + runcap;
    const int *run_len = run_p0 + runcap;
    const int *run_w = run_len + runcap;
    const int *run_tp = run_w + runcap;
    Unit U;
    U.nb = 0;
    int lo = 0, hi = nruns;  // last run with run_tp <= tile
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (run_tp[mid] <= tile) lo = mid; else hi = mid;
    }
    const int t_in = tile - run_tp[lo];
    U.w = run_w[lo];
    U.p0 = run_p0[lo] + t_in * TM;
    U.M = min(TM, run_len[lo] - t_in * TM);
    return U;
}

template <int TM>
__device__ __forceinline__ Unit decode_unit(const TmaKernelParams &k, const unsigned char *smem, int nruns,
                                            int64_t u) {
    const int *run_seg = reinterpret_cast<const int *>(smem + k.o_run);
    const int *run_p0 = run_seg + k.runcap;
    const int *run_len = run_p0 + k.runcap;
    const int *run_w = run_len + k.runcap;
    const int *run_tp = run_w + k.runcap;
    Unit U;
    const int tile = (int)(u / k.p.nsplit);
    U.nb = (int)(u % k.p.nsplit);
    int lo = 0, hi = nruns;  // last run with run_tp <= tile
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (run_tp[mid] <= tile) lo = mid; else hi = mid;
    }
    const int t_in = tile - run_tp[lo];
    U.w = run_w[lo];
    U.p0 = run_p0[lo] + t_in * TM;
    U.M = min(TM, run_len[lo] - t_in * TM);
    return U;
}

// This CTA's output columns for column block nb: whole 64-column blocks,
// counted from off[0], split over nsplit * CS parts.
__device__ __forceinline__ void column_range(const LoraParams &p, int nb, int q, int CS, int *n0, int *n1) {
    const int ntot = p.off[p.c] - p.off[0];
    const int nblk = (ntot + 63) / 64;
    const int parts = p.nsplit * CS;
    const int part = nb * CS + q;
    const int b0 = (int)((int64_t)part * nblk / parts), b1 = (int)((int64_t)(part + 1) * nblk / parts);
    *n0 = p.off[0] + 64 * b0;
    *n1 = min(p.off[p.c], p.off[0] + 64 * b1);
}

__device__ __forceinline__ int slice_at(const LoraParams &p, int col) {
    int j = 0;
    while (j + 1 < p.c && col >= p.off[j + 1]) ++j;
    return j;
}

// B rows of output columns [x0, x0 + rows) of slot w into dst (rows * R bf16,
// the layout of one box of tmB), completing on bar.  One tensor: one box of
// tmB.  Separate slice tensors: 64-row boxes, each from the slice its first
// column falls in (slice offsets and x0 are multiples of 64, so no box
// crosses a slice; columns past the last slice read rows that are not used).
__device__ __forceinline__ void load_b_rows(const TmaKernelParams &k, void *dst, int w, int x0, int rows,
                                            uint64_t *bar) {
    const LoraParams &p = k.p;
    if (!p.b_tuple) {
        tma_load_2d(dst, &k.tmB, 0, w * (int)p.N + x0, bar);
        return;
    }
    for (int r0 = 0; r0 < rows; r0 += 64) {
        const int col = x0 + r0;
        const int j = slice_at(p, col);
        tma_load_2d(static_cast<unsigned char *>(dst) + r0 * p.R * 2, &k.tmBs[j], 0,
                    w * p.b_rows[j] + p.b_row0[j] + (col - p.off[j]), bar);
    }
}

// Whether unit U is worked on at all; rank-0 slots have no work, invalid
// slots and ranks are reported.  Identical on every thread of the cluster.
__device__ __forceinline__ int unit_rank(const LoraParams &p, const Unit &U, bool report) {
    if (U.w < 0 || U.w >= p.max_loras) {
        if (report) atomicOr(p.status, CSGMV_STATUS_BAD_ADAPTER);
        return -1;
    }
    int r = p.lora_ranks[U.w];
    if (r < 0 || r > p.R) {
        if (report) atomicOr(p.status, CSGMV_STATUS_BAD_RANK);
        return -1;
    }
    return r;
}

// ---------------------------------------------------------------------------------- consumers
// bf16 hi / lo halves of a pair of fp32 values, packed for an mma A fragment.
__device__ __forceinline__ void split_pair(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
    hi = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
    lo = pack_bf16x2(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
}

// Expand of one unit on the 5th-generation tensor cores.  The tile's h (every
// slice) goes to shared memory as bf16 hi / lo operand tiles (128-byte rows,
// 128-byte swizzle); per 128-column stage warp 0 waits for the B tile, zeroes
// B's padding columns [r, round16(r)) if the rank is ragged, and one lane
// issues hi and lo tcgen05.mma per k16 step into one of two TMEM
// accumulators (a stage that crosses a slice boundary is split there).  Every
// warp then reads a 32-row x 32-column block of the accumulator (tcgen05.ld,
// its TMEM lane quarter), adds base from the staged tile in fp32 and stores
// 64-byte row pieces back through the permutation.  Warp 0 issues the next
// stage's MMAs before its own epilogue, so the tensor core runs ahead.
template <int TM, int MODE, typename IssueNext>
__device__ void expand_tc(const TmaKernelParams &k, unsigned char *smem, const Unit &U, int r, float sigma, int CS,
                          int n0, int n1, int nt, const int *tok, uint32_t tmem, uint32_t &ex_it, uint32_t &acc_it,
                          IssueNext issue_next) {
    static_assert(TM == 128, "the tensor-core expand takes 128-token tiles");
    const LoraParams &p = k.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (nt <= 0) return;
    Bars B = bars_of(k, smem);
    uint64_t *acc_full = reinterpret_cast<uint64_t *>(smem + k.o_tc);
    uint64_t *acc_empty = acc_full + 2;
    unsigned char *ah = smem + k.o_ah;
    const int RK = (r + 15) & ~15;
    const int ksteps = RK / 16;
    const int rpr = TM / CS;
    const float *hred = reinterpret_cast<const float *>(smem + k.o_hred);
    const int hp = k.hp;

    // h of every slice this CTA's columns touch (slices jfirst..): operand tile
    // 2(j - jfirst) (hi) and 2(j - jfirst) + 1 (lo), row m = token m of the
    // tile, columns [0, RK) of which [r, RK) are zero.
    const int jfirst = slice_at(p, n0);
    const int nsl = slice_at(p, n1 - 1) - jfirst + 1;
    if (nsl > k.ah_slices) {  // the launcher sized the tiles for fewer slices: refuse the unit
        if (tid == 0) atomicOr(p.status, kStatusTimeout);
        return;
    }
    const int cpr = RK / 8;
    const int per_slice = TM * cpr;
    for (int idx = tid; idx < nsl * per_slice; idx += kConsumerThreads) {
        const int jo = idx / per_slice, rem = idx % per_slice;
        const int j = jfirst + jo;
        const int m = rem / cpr, ch = rem % cpr;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int kk = ch * 8 + e;
            float x = 0.f;
            if (m < U.M && kk < r) {
                const int col = j * r + kk;
                if constexpr (MODE == kModeExpand) {
                    const int t = tok[m];
                    if (t >= 0)
                        x = p.h_f32 ? reinterpret_cast<const float *>(p.h)[(int64_t)t * p.ldh + col]
                                    : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col]);
                } else {
                    const int owner = m / rpr;
                    x = dsmem_ld_f32(dsmem_addr(hred + (m - owner * rpr) * hp + col, owner));
                }
            }
            v[e] = x;
        }
        uint4 hi, lo;
        split_pair(v[0], v[1], hi.x, lo.x);
        split_pair(v[2], v[3], hi.y, lo.y);
        split_pair(v[4], v[5], hi.z, lo.z);
        split_pair(v[6], v[7], hi.w, lo.w);
        const int off = m * 128 + ((ch ^ (m & 7)) << 4);
        *reinterpret_cast<uint4 *>(ah + (2 * jo) * kTcAhBytes + off) = hi;
        *reinterpret_cast<uint4 *>(ah + (2 * jo + 1) * kTcAhBytes + off) = lo;
    }
    fence_proxy_async_smem();  // the operand tiles are read by the tensor core
    __syncthreads();

    const uint32_t it0 = ex_it, a0 = acc_it;
    const int Rb = p.R * 2;  // bytes per B row (32, 64 or 128: its swizzle width)
    const int pcB = p.R / 8, shB = pc_shift_of(pcB);
    // MMAs of stage i (whole warp 0; one lane issues)
    auto mma_stage = [&](int i) {
        const uint32_t g = it0 + i;
        const int e = g % k.S2;
        mbar_wait(&B.ex_full[e], (g / k.S2) & 1, p.status, kStatusTimeout);
        unsigned char *bs = smem + k.o_ex + e * k.ex_stage + k.ex_b;
        if (RK != r) {  // B columns [r, RK) are adapter padding (even NaN): zero them
            const int c0 = r >> 3, nc = (RK >> 3) - c0;
            for (int idx = lane; idx < kTcCols * nc; idx += 32) {
                const int n = idx / nc, ch = c0 + idx % nc;
                uint16_t *q16 = reinterpret_cast<uint16_t *>(bs) + swz(n, ch, pcB, shB);
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2)
                    if (ch * 8 + e2 >= r) q16[e2] = 0;
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const uint32_t ga = a0 + i;
        const int a = ga & 1;
        mbar_wait(&acc_empty[a], ((ga >> 1) & 1) ^ 1, p.status, kStatusTimeout);
        tc_fence_after();
        if (lane == 0) {
            const int x0 = n0 + i * kTcCols;
            const int ncols = min(n1, x0 + kTcCols) - x0;  // a multiple of 16
            const uint32_t bsa = smem_u32(bs);
            int c0 = 0;
            while (c0 < ncols) {
                const int j = slice_at(p, x0 + c0);
                const int c1 = j + 1 < p.c ? min(ncols, p.off[j + 1] - x0) : ncols;
                const uint32_t idesc = idesc_bf16_f32(128, c1 - c0);
                const uint32_t d = tmem + (uint32_t)(a * kTcCols + c0);
                const int jo = j - jfirst;
                const uint32_t ahi = smem_u32(ah + (2 * jo) * kTcAhBytes), alo = smem_u32(ah + (2 * jo + 1) * kTcAhBytes);
                for (int ks = 0; ks < ksteps; ++ks) {
                    const uint64_t bd = smem_desc_kmajor(bsa + (uint32_t)(c0 * Rb + ks * 32), Rb);
                    tc_mma_bf16(d, smem_desc_kmajor(ahi + ks * 32, 128), bd, idesc, ks > 0);
                    tc_mma_bf16(d, smem_desc_kmajor(alo + ks * 32, 128), bd, idesc, true);
                }
                c0 = c1;
            }
            tc_commit(&acc_full[a]);
        }
        __syncwarp();
    };

    if (warp == 0) mma_stage(0);
    const int quarter = warp & 3, cg = warp >> 2;  // TMEM lanes 32*quarter.., columns 32*cg..
    for (int i = 0; i < nt; ++i) {
        issue_next(i);
        if (warp == 0 && i + 1 < nt) mma_stage(i + 1);
        const uint32_t g = it0 + i;
        const int e = g % k.S2;
        const uint32_t ga = a0 + i;
        const int a = ga & 1;
        mbar_wait(&acc_full[a], (ga >> 1) & 1, p.status, kStatusTimeout);
        mbar_wait(&B.ex_full[e], (g / k.S2) & 1, p.status, kStatusTimeout);
        tc_fence_after();
        __syncwarp();  // tcgen05.ld is warp-wide
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(a * kTcCols + 32 * cg), v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
        unsigned char *ys = smem + k.o_ex + e * k.ex_stage;
        const int x0 = n0 + i * kTcCols, x1 = min(n1, x0 + kTcCols);
        const int row = 32 * quarter + lane;
        if (row < U.M) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int lc = 32 * cg + 8 * c4;
                if (x0 + lc < x1) {
                    uint4 *ptr = reinterpret_cast<uint4 *>(ys + (lc >> 6) * TM * 128 + row * 128 +
                                                           ((((lc & 63) >> 3) ^ (row & 7)) << 4));
                    uint4 bv = p.accumulate ? *ptr : make_uint4(0, 0, 0, 0);
                    float2 f;
                    f = unpack_bf16x2(bv.x); bv.x = pack_bf16x2(f.x + sigma * v[8 * c4 + 0], f.y + sigma * v[8 * c4 + 1]);
                    f = unpack_bf16x2(bv.y); bv.y = pack_bf16x2(f.x + sigma * v[8 * c4 + 2], f.y + sigma * v[8 * c4 + 3]);
                    f = unpack_bf16x2(bv.z); bv.z = pack_bf16x2(f.x + sigma * v[8 * c4 + 4], f.y + sigma * v[8 * c4 + 5]);
                    f = unpack_bf16x2(bv.w); bv.w = pack_bf16x2(f.x + sigma * v[8 * c4 + 6], f.y + sigma * v[8 * c4 + 7]);
                    *ptr = bv;
                }
            }
        }
        __syncwarp();
        // this warp's 32 rows x 32 columns, 64-byte row pieces
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int idx = lane + 32 * it, rr = idx >> 2, c4 = idx & 3;
            const int row2 = 32 * quarter + rr, lc = 32 * cg + 8 * c4, col = x0 + lc;
            if (row2 < U.M && col < x1) {
                const int t = tok[row2];
                if (t >= 0)
                    *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) = *reinterpret_cast<const uint4 *>(
                        ys + (lc >> 6) * TM * 128 + row2 * 128 + ((((lc & 63) >> 3) ^ (row2 & 7)) << 4));
            }
        }
        fence_proxy_async_smem();  // the in-place epilogue writes before a TMA refills the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.ex_empty[e]);
    }
    ex_it += nt;
    acc_it += nt;
}

// The sixteen warps gather the permuted x / base rows with coalesced
// 16-byte cp.async (completion folded into the stage's mbarrier), run the
// tensor-core math and the epilogue, and write y back with 16-byte stores.
template <int TM, int RMAX, int MODE, bool TC>
__device__ void consumer_loop(const TmaKernelParams &k, unsigned char *smem, int q, int CS, int nruns,
                              int64_t nunits, int cid, int ncl, uint32_t tmem) {
    using G = Geo<TM, TC>;
    constexpr int SHT = (3 * RMAX / 8 + G::WN - 1) / G::WN;  // shrink n8 tiles per warp (c <= 3)
    constexpr int KS = RMAX / 16;                             // expand k16 steps at most
    const LoraParams &p = k.p;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp / G::WN, wn = warp % G::WN;
    Bars B = bars_of(k, smem);
    int *tokb = reinterpret_cast<int *>(smem + k.o_tok);
    const int cR = p.c * p.R;
    float *hpart = reinterpret_cast<float *>(smem + k.o_hpart);
    float *hred = reinterpret_cast<float *>(smem + k.o_hred);
    const int hp = k.hp;
    const int nkc = (int)((p.K + 63) / 64);
    const int kc0 = (int)((int64_t)q * nkc / CS), kc1 = (int)((int64_t)(q + 1) * nkc / CS);
    const int rpr = TM / CS;  // rows of the reduction owned by each CTA
    uint32_t sh_is = 0, sh_it = 0, ex_is = 0, ex_it = 0;
    uint32_t acc_it = 0;  // tensor-core expand: stages whose accumulator was used

    for (int64_t u = cid; u < nunits; u += ncl) {
        const Unit U = decode_unit<TM>(k, smem, nruns, u);
        const int r = unit_rank(p, U, q == 0 && tid == 0);
        if (r < 0) continue;
        if (r == 0) {
            // shrink: zero h rows; non-accumulating expand: zero output rows
            if constexpr (MODE == kModeShrink) {
                const int cR = p.c * p.R;
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
                    int n0, n1;
                    column_range(p, U.nb, q, CS, &n0, &n1);
                    const int nch = (n1 - n0) / 8;
                    for (int m = 0; m < U.M; ++m) {
                        const int t = p.permutation[U.p0 + m];
                        if (t < 0 || t >= p.num_tokens) continue;
                        for (int ch = tid; ch < nch; ch += kConsumerThreads)
                            *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + n0 + 8 * ch) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            continue;
        }
        const float sigma = p.scalings[U.w];
        // token list of the tile (the permutation slice), shared by all warps
        int *tok = tokb;
        fence_proxy_async_smem();  // this thread's generic writes before TMA copies reuse the memory
        __syncthreads();  // every warp is done with the previous unit's list
        for (int m = tid; m < TM; m += kConsumerThreads) {
            int t = -1;
            if (m < U.M) {
                t = p.permutation[U.p0 + m];
                if (t < 0 || t >= p.num_tokens) { atomicOr(p.status, CSGMV_STATUS_BAD_PERMUTATION); t = -1; }
            }
            tok[m] = t;
        }
        __syncthreads();
        // A tile of consecutive tokens (the usual prefill case: one request's
        // tokens in order) loads its x and base rows as TMA boxes instead of
        // row gathers.  Rows past the tile in the box are read, never used.
        bool rows_tma = false;
        if constexpr (TM == 128) {
            bool mine = true;
            const int t0 = tok[0];
            for (int m = tid; m < U.M; m += kConsumerThreads) mine = mine && tok[m] == t0 + m;
            rows_tma = __syncthreads_and(mine && t0 >= 0 && k.row_tma) != 0;
        }
        const int cr = p.c * r;
        const int crp = (cr + 7) & ~7;
        const int ksteps = (r + 15) / 16;
        const int nch = MODE != kModeExpand ? kc1 - kc0 : 0;
        int nt = 0, n0 = 0, n1 = 0;
        if constexpr (MODE != kModeShrink) {
            column_range(p, U.nb, q, CS, &n0, &n1);
            nt = n1 > n0 ? (n1 - n0 + G::NT - 1) / G::NT : 0;
        }

        // x rows of K chunk `ci` of this unit into the next shrink stage
        auto issue_x = [&](int ci) {
            const int s = sh_is % k.S1;
            mbar_wait(&B.sh_empty[s], ((sh_is / k.S1) & 1) ^ 1, p.status, kStatusTimeout);
            __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(smem + k.o_sh + s * k.sh_stage);
            const int64_t k0 = (int64_t)(kc0 + ci) * 64;
            if (tid == 0) {  // the A rows of this chunk: one TMA box (and the x rows: another)
                mbar_arrive_expect_tx(&B.sh_full[s], k.a_rows * 128 + (rows_tma ? TM * 128 : 0));
                tma_load_2d(smem + k.o_sh + s * k.sh_stage + k.sh_a, &k.tmA, (int)k0, U.w * cR, &B.sh_full[s]);
                if (rows_tma) tma_load_2d(xs, &k.tmX, (int)k0, tok[0], &B.sh_full[s]);
            }
            if (!rows_tma)
            for (int idx = tid; idx < U.M * 8; idx += kConsumerThreads) {
                const int m = idx >> 3, ch = idx & 7;
                const int t = tok[m];
                const int64_t kk = k0 + ch * 8;
                const bool ok = t >= 0 && kk < p.K;
                cp_async16(xs + swz(m, ch, 8, 0), ok ? p.x + (int64_t)t * p.K + kk : p.x, ok ? 16 : 0);
            }
            cp_async_mbar_arrive(&B.sh_full[s]);
            ++sh_is;
        };
        // base rows of column tile `i` into the next expand stage
        auto issue_base = [&](int i) {
            const int e = ex_is % k.S2;
            mbar_wait(&B.ex_empty[e], ((ex_is / k.S2) & 1) ^ 1, p.status, kStatusTimeout);
            unsigned char *ys = smem + k.o_ex + e * k.ex_stage;
            const int x0 = n0 + i * G::NT, x1 = min(n1, x0 + G::NT);
            const bool base_tma = rows_tma && p.accumulate;
            if (tid == 0) {  // the B rows of this column tile: one TMA box (base rows: NB64 more)
                mbar_arrive_expect_tx(&B.ex_full[e], G::NT * p.R * 2 + (base_tma ? G::NB64 * TM * 128 : 0));
                load_b_rows(k, ys + k.ex_b, U.w, x0, G::NT, &B.ex_full[e]);
                if (base_tma)
                    for (int bx = 0; bx < G::NB64; ++bx)
                        tma_load_2d(ys + bx * TM * 128, &k.tmY, x0 + 64 * bx, tok[0], &B.ex_full[e]);
            }
            if (p.accumulate && !base_tma) {
                for (int idx = tid; idx < U.M * (G::NT / 8); idx += kConsumerThreads) {
                    const int m = idx / (G::NT / 8), c8 = idx % (G::NT / 8);
                    const int col = x0 + 8 * c8;
                    const int t = tok[m];
                    if (t >= 0 && col < x1)
                        cp_async16(ys + (c8 >> 3) * TM * 128 + m * 128 + (((c8 & 7) ^ (m & 7)) << 4),
                                   p.y + (int64_t)t * p.N + col, 16);
                }
            }
            cp_async_mbar_arrive(&B.ex_full[e]);
            ++ex_is;
        };

        // Everything that does not depend on h goes out first: the first
        // shrink stages and the first expand stages.
        const int sh_pre = min(nch, k.S1 - 1);
        for (int ci = 0; ci < sh_pre; ++ci) issue_x(ci);
        const int ex_pre = min(nt, k.S2 - 1);
        for (int i = 0; i < ex_pre; ++i) issue_base(i);

        if constexpr (MODE != kModeExpand) {
            // ---------------------------------------------------------------- shrink
            float acc[SHT][4];
#pragma unroll
            for (int i = 0; i < SHT; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
            for (int ci = 0; ci < nch; ++ci) {
                if (ci + k.S1 - 1 < nch) issue_x(ci + k.S1 - 1);
                const int s = sh_it % k.S1;
                mbar_wait(&B.sh_full[s], (sh_it / k.S1) & 1, p.status, kStatusTimeout);
                const __nv_bfloat16 *xs = reinterpret_cast<const __nv_bfloat16 *>(smem + k.o_sh + s * k.sh_stage);
                const __nv_bfloat16 *as = reinterpret_cast<const __nv_bfloat16 *>(smem + k.o_sh + s * k.sh_stage + k.sh_a);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    uint32_t a[4];
                    ldmatrix_x4(a[0], a[1], a[2], a[3], xs + swz(wm * 16 + (lane & 15), 2 * ks + (lane >> 4), 8, 0));
#pragma unroll
                    for (int i = 0; i < SHT; ++i) {
                        const int j = wn + G::WN * i;
                        if (j * 8 < crp) {
                            uint32_t b0, b1;
                            ldmatrix_x2(b0, b1, as + swz(j * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1), 8, 0));
                            mma_bf16_16816(acc[i], a, b0, b1);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.sh_empty[s]);
                ++sh_it;
            }
            __syncthreads();  // the partials alias the shrink ring: every warp must be done with it
#pragma unroll
            for (int i = 0; i < SHT; ++i) {
                const int j = wn + G::WN * i;
                if (j * 8 < crp) {
                    const int row = wm * 16 + (lane >> 2), col = j * 8 + 2 * (lane & 3);
                    *reinterpret_cast<float2 *>(hpart + row * hp + col) = make_float2(acc[i][0], acc[i][1]);
                    *reinterpret_cast<float2 *>(hpart + (row + 8) * hp + col) = make_float2(acc[i][2], acc[i][3]);
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
                    // every peer's partial is loaded before any is summed, so the
                    // distributed-shared-memory loads overlap (clusters of up to 8 CTAs)
                    float4 t4[8];
#pragma unroll
                    for (int peer = 0; peer < 8; ++peer)
                        if (peer < CS) t4[peer] = dsmem_ld_f4(dsmem_addr(hpart + row * hp + 4 * v, peer));
                    float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int peer = 0; peer < 8; ++peer)
                        if (peer < CS) { s4.x += t4[peer].x; s4.y += t4[peer].y; s4.z += t4[peer].z; s4.w += t4[peer].w; }
                    *reinterpret_cast<float4 *>(hred + rr * hp + 4 * v) = s4;
                }
                cluster_arrive();
                cluster_wait();
            } else {
                named_bar_sync(kBarConsumers, kConsumerThreads);
            }
            if constexpr (MODE == kModeShrink) {
                const float *src = CS > 1 ? hred : hpart;
                const int row0 = CS > 1 ? q * rpr : 0;
                const int nrows = CS > 1 ? rpr : TM;
                const int cR = p.c * p.R;
                for (int idx = tid; idx < nrows * cR; idx += kConsumerThreads) {
                    const int rr = idx / cR, col = idx % cR;
                    const int row = row0 + rr;
                    if (row >= U.M) continue;
                    const int t = tok[row];
                    if (t < 0) continue;
                    const float v = col < cr ? src[rr * hp + col] : 0.f;
                    if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = v;
                    else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(v);
                }
            }
        }

        if constexpr (MODE != kModeShrink && TC) {
            expand_tc<TM, MODE>(k, smem, U, r, sigma, CS, n0, n1, nt, tok, tmem, ex_it, acc_it, [&](int i) {
                if (i + k.S2 - 1 < nt) issue_base(i + k.S2 - 1);
            });
        } else if constexpr (MODE != kModeShrink) {
            // ---------------------------------------------------------------- expand
            const int rowA = wm * 16 + (lane >> 2), rowB = rowA + 8;
            // h fragments (bf16 hi / lo pairs) of one slice for this warp's 16 rows
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
                    if (CS > 1) {
                        const int owner = row / rpr;
                        return dsmem_ld_f32(dsmem_addr(hred + (row - owner * rpr) * hp + col, owner));
                    }
                    return hpart[row * hp + col];
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
            for (int i = 0; i < nt; ++i) {
                if (i + k.S2 - 1 < nt) issue_base(i + k.S2 - 1);
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
                    // Slices this warp's columns touch (one, unless a slice
                    // boundary falls inside them); each n8 tile uses its own.
                    const int jl = slice_at(p, wc0), jh = slice_at(p, min(wc0 + G::WCOLS, x1) - 1);
                    for (int jj = jl; jj <= jh; ++jj) {
                        if (jj != cur) load_slice(jj);
#pragma unroll
                        for (int t8 = 0; t8 < G::EXT; t8 += 2) {
                            const int lc = wn * G::WCOLS + 8 * t8;  // stage-local column of tile t8
                            if (x0 + lc >= x1) continue;
                            const bool use0 = jl == jh || slice_at(p, x0 + lc) == jj;
                            const bool use1 = x0 + lc + 8 < x1 && (jl == jh || slice_at(p, x0 + lc + 8) == jj);
#pragma unroll
                            for (int ks = 0; ks < KS; ++ks) {
                                if (ks < ksteps) {
                                    uint32_t b00, b01, b10, b11;
                                    if (RMAX == 16 && p.R == 8) {
                                        const int nrow = lc + 8 * ((lane >> 3) & 1) + (lane & 7);
                                        ldmatrix_x2(b00, b10, bs + nrow * 8);
                                        b01 = 0u;
                                        b11 = 0u;
                                    } else {
                                        const int nrow = lc + 8 * (lane >> 4) + (lane & 7);
                                        const int ch = 2 * ks + ((lane >> 3) & 1);
                                        ldmatrix_x4(b00, b01, b10, b11, bs + swz(nrow, ch, pcB, shB));
                                    }
                                    if (use0) {
                                        mma_bf16_16816(acc[t8], fhi[ks], b00, b01);
                                        mma_bf16_16816(acc[t8], flo[ks], b00, b01);
                                    }
                                    if (use1) {
                                        mma_bf16_16816(acc[t8 + 1], fhi[ks], b10, b11);
                                        mma_bf16_16816(acc[t8 + 1], flo[ks], b10, b11);
                                    }
                                }
                            }
                        }
                    }
                }
                // y = base + sigma * acc, in place in the staged base tile
#pragma unroll
                for (int t8 = 0; t8 < G::EXT; ++t8) {
                    const int lc = wn * G::WCOLS + 8 * t8 + 2 * (lane & 3);
                    if (x0 + wn * G::WCOLS + 8 * t8 >= x1) continue;
                    const int bx = lc >> 6, cb = lc & 63;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int row = hh ? rowB : rowA;
                        if (row >= U.M) continue;
                        uint32_t *ptr = reinterpret_cast<uint32_t *>(ys + bx * TM * 128 + row * 128 +
                                                                     ((((cb >> 3) ^ (row & 7))) << 4) + (cb & 7) * 2);
                        const float2 bv = p.accumulate ? unpack_bf16x2(*ptr) : make_float2(0.f, 0.f);
                        *ptr = pack_bf16x2(bv.x + sigma * acc[t8][2 * hh], bv.y + sigma * acc[t8][2 * hh + 1]);
                    }
                }
                __syncwarp();
                // this warp's 16 rows x WCOLS columns go out as 16-byte stores
                constexpr int CPR = G::WCOLS / 8;  // 16-byte chunks per row
                for (int idx = lane; idx < 16 * CPR; idx += 32) {
                    const int row = wm * 16 + idx / CPR;
                    const int lc = wn * G::WCOLS + 8 * (idx % CPR);
                    const int col = x0 + lc;
                    if (row >= U.M || col >= x1) continue;
                    const int t = tok[row];
                    if (t < 0) continue;
                    const int bx = lc >> 6, c8 = (lc & 63) >> 3;
                    *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) =
                        *reinterpret_cast<const uint4 *>(ys + bx * TM * 128 + row * 128 + ((c8 ^ (row & 7)) << 4));
                }
                fence_proxy_async_smem();  // the in-place epilogue writes before a TMA refills the stage
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.ex_empty[e]);
                ++ex_it;
            }
        }
    }
}

template <int TM, int RMAX, int MODE, bool TC>
__global__ void __launch_bounds__(kTmaThreads, 1) lora_tma_kernel(const __grid_constant__ TmaKernelParams k) {
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
        Bars B = bars_of(k, smem);
        for (int i = 0; i < k.S1; ++i) { mbar_init(&B.sh_full[i], 1 + kConsumerThreads); mbar_init(&B.sh_empty[i], kConsumerWarps); }
        for (int i = 0; i < k.S2; ++i) { mbar_init(&B.ex_full[i], 1 + kConsumerThreads); mbar_init(&B.ex_empty[i], kConsumerWarps); }
        if constexpr (TC) {
            uint64_t *acc = reinterpret_cast<uint64_t *>(smem + k.o_tc);
            for (int i = 0; i < 2; ++i) { mbar_init(&acc[i], 1); mbar_init(&acc[2 + i], kConsumerWarps); }
        }
        fence_mbar_init();
        prefetch_tmap(&k.tmA);
        prefetch_tmap(&k.tmB);
        if (k.p.b_tuple)
            for (int j = 0; j < kMaxSlices; ++j) prefetch_tmap(&k.tmBs[j]);
        if (k.row_tma) {
            prefetch_tmap(&k.tmX);
            prefetch_tmap(&k.tmY);
        }
    }
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + k.o_tc + 32);
    if constexpr (TC) {
        if (threadIdx.x < 32) {  // one warp owns the TMEM accumulators of the CTA
            tmem_alloc(tmem_slot, kTcTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    int nruns = 0;
    const int ntiles = build_run_table<TM>(k, smem, &nruns);  // ends with __syncthreads
    uint32_t tmem = 0;
    if constexpr (TC) {
        tc_fence_after();
        tmem = *tmem_slot;
    }
    const int64_t nunits = (int64_t)ntiles * k.p.nsplit;
    const int cid = blockIdx.x / CS, ncl = gridDim.x / CS;
    consumer_loop<TM, RMAX, MODE, TC>(k, smem, q, CS, nruns, nunits, cid, ncl, tmem);
    if constexpr (MODE != kModeExpand) {
        if (CS > 1) {  // peers may still read this CTA's shared memory
            cluster_arrive();
            cluster_wait();
        }
    }
    if constexpr (TC) {  // every epilogue has read its accumulator
        tc_fence_before();
        __syncthreads();
        if (threadIdx.x < 32) {
            tc_fence_after();
            tmem_dealloc(tmem, kTcTmemCols);
        }
    }
}

}  // namespace csgmv
