// Streaming tcgen05 expand for 128-token tiles (sglang chunked_backend.py
// run_lora_b_sgemm, and the expand half of run_qkv_lora / run_gate_up_lora
// when h comes from a workspace; shapes from base_backend.py):
//     y[t][n] = (accumulate ? y[t][n] : 0) + sigma_w * sum_{k<r} h[t][j*r + k] * B_j[w][n][k]
// for every token t of a tile on slot w, and n in slice j.
//
// The expand is a read-modify-write stream of base: a prefill batch moves
// gigabytes of base rows against kilobytes of h and megabytes of B, so the
// kernel is built to keep HBM busy.  One CTA per SM walks its units (a tile of
// up to 128 tokens of one slot x a block of columns inside one slice) with a
// fixed stride; every role runs the same unit walk and the roles are linked
// only by mbarriers, so loads of later stages and units stream while earlier
// ones are multiplied and written back:
//   warp 0      base producer: per stage of kStCols columns, the tile's base
//               rows (128-row TMA boxes when the tile's tokens are
//               consecutive, else TMA 4-row gathers) into a ring of base
//               slots;
//   warp 2      B producer: per stage, the slot's B rows (one TMA box per 64
//               columns) into a ring of B slots, running ahead of the rest;
//   warp 1      MMA issuer: per stage, y_delta = h B^T on the tensor cores
//               (h as a bf16 hi + lo pair, so it keeps ~16 bits) into one of
//               kStAcc TMEM accumulators; completions free the B slot;
//   warps 4-7   operands: per unit, the token list and h of the unit's slice
//               from global memory as bf16 hi / lo pairs written into TMEM
//               (each warp its lane quarter), where the MMA takes them as its A
//               operand; double-buffered one unit ahead;
//   warps 8..   epilogue, teams of four warps that take the stages in turn: each
//               warp reads its 32 accumulator rows (tcgen05.ld), adds base in
//               fp32 and writes the rounded rows back in place, then stores
//               its 32-row piece with TMA box stores (a full tile of
//               consecutive tokens) or 16-byte row stores through the token
//               list; a base slot is handed back once its stores have read it.
// Every wait is bounded; on a timeout the kernel sets a status bit and ends.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kStTeams = 2;              // epilogue teams of four warps, taking stages in turn
constexpr int kStOpWarp0 = 4;            // four operand warps, one TMEM lane quarter each
constexpr int kStEpiWarp0 = 8;
constexpr int kStEpiWarps = 4 * kStTeams;
constexpr int kStWarps = kStEpiWarp0 + kStEpiWarps;
constexpr int kStThreads = kStWarps * 32;
constexpr int kStBoxes = 1;              // 64-column boxes per stage
constexpr int kStCols = 64 * kStBoxes;   // output columns per stage
constexpr int kStTmemCols = 512;         // the allocation: a power of two
// h of a unit in TMEM as the MMA's A operand: rows in lanes, two bf16 of
// consecutive K per 32-bit column; the hi half in columns [0, 32) and the lo
// half in [32, 64) of an operand buffer, two buffers at the top of TMEM.
constexpr int kStOpCols = 64;
constexpr int kStOpCol0 = kStTmemCols - 2 * kStOpCols;
// TMEM accumulators of kStCols columns below the operand buffers.  Every
// mbarrier of the epilogue is waited on by one team only: stage g takes
// accumulator g % kStAcc, base slot g % Sy and team g % kStTeams, so kStAcc
// and Sy are multiples of kStTeams (a team that waited on a barrier another
// team also waits on could take a phase two completions old for the current
// one).
constexpr int kStAcc = (kStOpCol0 / kStCols) / kStTeams * kStTeams;
constexpr int kStTileBytes = 128 * 128;  // 128 rows x 64 bf16: one base box
constexpr int kStBSlots = 6;             // B tiles in flight (needed only until their MMAs are done)
static_assert(kStAcc >= kStTeams, "every team needs an accumulator");

// Base rows of a tile of consecutive tokens move as TMA boxes of 128, 64, 32,
// 16 and 8 rows (one tensor map each), so that a tile of M < 128 tokens loads
// round8(M) rows rather than 128.  (The same for the shrink's x rows measured
// slower: 112 -> 141 us on the prefill shrink.)
constexpr int kRowBoxLevels = 5;

#ifdef __CUDACC__
// Rows [0, M) (M <= 128) of the consecutive tokens t0, t0 + 1, ..., columns
// [x, x + 64), into a 128-byte-swizzled tile of 128-byte rows at dst: M
// rounded up to 8 as a sum of the box heights, largest first (every box
// starts on an 8-row, i.e. 1024-byte, boundary).  Returns the bytes loaded.
__device__ __forceinline__ uint32_t load_row_boxes(void *dst, const CUtensorMap *maps, int x, int t0, int M,
                                                   uint64_t *bar) {
    const int Mr = (M + 7) & ~7;
    int o = 0;
#pragma unroll
    for (int l = 0; l < kRowBoxLevels; ++l) {
        const int h = 128 >> l;
        if (Mr - o >= h) {
            tma_load_2d(static_cast<unsigned char *>(dst) + o * 128, &maps[l], x, t0 + o, bar);
            o += h;
        }
    }
    return (uint32_t)Mr * 128;
}
__device__ __forceinline__ uint32_t row_box_bytes(int M) { return (uint32_t)((M + 7) & ~7) * 128; }
#endif

struct StreamParams {
    CUtensorMap tmB[kMaxSlices];  // slice j of B: L * b_rows[j] rows of R bf16, box R x 64
    CUtensorMap tmY[kRowBoxLevels];  // base / y (s rows, N): boxes 64 x (128 >> l), 128-byte swizzle (loads)
    CUtensorMap tmYs;             // the same, box 64 x 32 (one epilogue warp's store)
    CUtensorMap tmYg;             // the same, box 64 x 1 (4-row gathers)
    LoraParams p;
    int runcap, max_segments;
    int cb;                       // columns of a unit (multiple of 64)
    int upt;                      // units per tile: sum over slices of ceil(width / cb)
    int Sy, Sb;                   // base slots, B slots
    int o_bar, o_run, o_tok, o_yring, o_bring;
    int y_slot_bytes, b_slot_bytes;  // kStBoxes base boxes; kStCols rows of B
};

// Streaming tcgen05 shrink for 128-token tiles (run_lora_a_sgemm):
//     h[t][j*r + k] = sum_i x[t][i] * A[w][j*r + k][i]
// One CTA per SM walks its units (a tile of up to 128 tokens of one slot x
// one of P parts of K) with a fixed stride:
//   warp 0      producer: the tile's token list, then per 64-wide K chunk the
//               x rows (one 128-row TMA box for consecutive tokens, else 32
//               TMA 4-row gathers) and the slot's A rows [0, round16(c*r)) as
//               16-row boxes, into a ring of S stages;
//   warp 1      MMA issuer: h_part = x A^T over the unit's K chunks into one of
//               two TMEM accumulators (the next unit's MMAs run while the last
//               one is written out);
//   warps 2-5   epilogue: each warp its 32 rows of the accumulator
//               (tcgen05.ld), written as fp32 (or bf16) h rows.
// The part count P is chosen on the device from the exact tile count (the
// best-filled last wave, at most max_parts).  With P > 1 (the csgmv_qkv
// workspace path) part p of K goes to plane p of the workspace, P is written
// to the workspace header, and the expand sums the planes in order; P = 1
// writes h itself, with zeros in columns [c*r, c*R) and in rows of rank-0
// tokens.
constexpr int kShWarps = 6;
// 64-column K chunks per ring stage (at most; the launcher takes three when
// three stages of them fit, else two): the x boxes of a stage are
// neighbouring 128-byte pieces of each token row, which the DRAM serves far
// better asked for together (a probe streaming x-shaped rows: 5.0 TB/s with
// one chunk per request, 6.1 TB/s with two, 6.6 TB/s with four, for the same
// bytes in flight).
constexpr int kShChunksMax = 3;
constexpr int kShThreads = kShWarps * 32;
constexpr int kShEpiWarp0 = 2;

struct ShrinkParams {
    CUtensorMap tmX;   // x (s rows, K): box 64 x 128, 128-byte swizzle
    CUtensorMap tmXg;  // the same, box 64 x 1 (4-row gathers)
    CUtensorMap tmXp[4];  // the same, boxes of 64, 32, 16 and 8 rows (partial tiles: one box, little overfetch)
    CUtensorMap tmA;   // A (L * c * R rows, K): box 64 x 16, 128-byte swizzle
    CUtensorMap tmA32, tmA64;  // the same, boxes of 32 and 64 rows (fewer TMA instructions per stage)
    // 3-D views (64 columns, rows, K chunks of 64) of x and A whose box holds
    // a stage's `chunks` chunks in one instruction: x 128 rows, A round16(c*R)
    // rows, written [chunk][row][128 B] like the per-chunk tiles (use3d: K is
    // a multiple of 64 and both maps encoded)
    CUtensorMap tmX3, tmA3;
    CUtensorMap tmA3s[3];  // the A view with boxes of 16, 32 and 64 rows (a slot whose c*r needs fewer rows)
    int use3d;
    LoraParams p;
    int runcap, max_segments;
    int max_parts;     // parts of K the output holds (1: h itself)
    int *parts_out;    // where the chosen part count goes (the workspace header), or NULL
    int S;             // ring stages
    int o_bar, o_run, o_tok, o_ring;
    int chunks;        // K chunks per stage (1 .. kShChunksMax)
    int stage_bytes;   // `chunks` x tiles, then `chunks` A tiles of round16(c * R) rows
    int a_off;         // offset of the first A tile in a stage (`chunks` x tiles)
    int a_bytes;       // bytes of one A tile
    int64_t plane;     // elements of h between two parts (P > 1)
};

}  // namespace csgmv
