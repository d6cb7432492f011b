// Decode-shaped csgmv_qkv with an h workspace: a split-K shrink kernel and an
// expand kernel, neither using thread-block clusters (sglang chunked_backend.py
// run_qkv_lora / run_gate_up_lora over run_lora_a_sgemm + run_lora_b_sgemm;
// shapes from base_backend.py).
//
// A decode batch is a few tokens per slot, so a call is a chain of short
// dependent steps, not a stream: its time is launch, table, first-byte
// latency and the per-SM copy rate, and a cluster barrier alone costs more
// than the arithmetic.  Both kernels therefore:
//   - derive the tile table in one round of loads (segments, slot ranks and
//     scalings, and the whole permutation, all before any of them is used);
//   - put every copy of a unit in flight at once, spread over the warps;
//   - cut the work into about one unit per SM.
// Shrink: unit = (tile, part of K).  The tile's x rows (one bulk copy per
// token) and the slot's A rows (one 64-column TMA box per K chunk) land on
// one mbarrier; mma.sync m16n8k16 with fp32 accumulators; the partial sums go
// to plane `part` of the workspace, rows indexed by sorted position.
// Expand: unit = (tile, block of output columns of one slice).  Launched as a
// programmatic dependent of the shrink, it loads its base rows and B rows
// while the shrink is still running, then waits for the shrink, sums the
// planes of its slice's h columns in part order (deterministic) straight into
// mma A fragments (h as a bf16 hi + lo pair), runs the MMAs per 16-column
// pair and stores y = base + sigma h B^T from registers.
// The inner loops are specialised on warp-uniform tile counts and address
// shared memory through precomputed 32-bit offsets: with a handful of
// tokens per tile, instruction issue, not memory, sets the pace of a warp.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kDecThreads = 256;     // shrink CTA
constexpr int kDecWarps = kDecThreads / 32;
// expand CTA: 16 warps at 64 registers, so that it shares an SM with the
// shrink (256 threads at 128 registers); one plane-sum item per thread
constexpr int kDecExpThreads = 512;
constexpr int kDecExpItems = 1;
constexpr int kDecExpWarps = kDecExpThreads / 32;
constexpr int kDecSegCap = 512;      // segments (max_segments) the kernels take
constexpr int kDecLoraCap = 256;    // slots (max_loras)
constexpr int kDecRecCap = 256;     // tile records of the batch info's table loaded up front
constexpr int kDecPartsTarget = 16; // parts of K per tile at most (one batch of plane loads in the expand)

// Shared-memory table (ints): seg_indptr, weight_indices, slot ranks and
// scalings, the permutation, the run table, then the first records of the
// batch info's tile table.
constexpr int kDecTabIp = 0;
constexpr int kDecTabSw = kDecTabIp + kDecSegCap + 1;
constexpr int kDecTabRk = kDecTabSw + kDecSegCap;
constexpr int kDecTabSc = kDecTabRk + kDecLoraCap;
constexpr int kDecTabPerm = kDecTabSc + kDecLoraCap;
constexpr int kDecTabRunW = kDecTabPerm + kDecPermCap;
constexpr int kDecTabRunP0 = kDecTabRunW + kDecSegCap;
constexpr int kDecTabRunN = kDecTabRunP0 + kDecSegCap;
constexpr int kDecTabRunT0 = kDecTabRunN + kDecSegCap;
constexpr int kDecTabScratch = kDecTabRunT0 + kDecSegCap + 1;
constexpr int kDecTabRec = kDecTabScratch + 32;  // records of the batch info's tile table
constexpr int kDecTabInts = kDecTabRec + 4 * kDecRecCap;

struct DecodeParams {
    CUtensorMap tmA;               // A (L*c*R rows, K): box 64 x a_rows, 128-byte swizzle
    CUtensorMap tmB;               // B (L*N rows, R): box R x 64, swizzle of the R*2-byte row
    CUtensorMap tmBs[kMaxSlices];  // B per slice tensor (p.b_tuple): box R x 64
    // p.h: the fp32 planes, p.h_plane floats apart, p.h_parts of them held
    // by the workspace; plane rows are sorted positions, p.ldh floats each
    LoraParams p;
    int max_segments;
    int tile_cap;     // records the batch info's tile table holds
    int nkc;          // 64-column chunks of K
    int shrink_grid;  // CTAs of the shrink launch: both kernels derive the part count from it
    int kc_max;       // shrink: K chunks staged per pass
    int a_rows;       // shrink: rows of one A box (round16(c*R))
    int xpitch;       // shrink: bytes per staged x row
    int cols_max;     // expand: output columns of one unit at most (a multiple of 64)
    int ypitch;       // expand: bytes per staged base row
    int o_bar, o_tab, o_a, o_x, o_y, o_b, o_h;  // shared-memory offsets
};

}  // namespace csgmv
