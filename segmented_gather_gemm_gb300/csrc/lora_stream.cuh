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
//   warp 0      producer: per 64-column stage, the slot's B rows (one TMA
//               box) and the tile's base rows (one 128-row TMA box when the
//               tile's tokens are consecutive, else 32 TMA 4-row gathers)
//               into a ring of S slots;
//   warp 1      MMA issuer: per stage, y_delta = h B^T on the tensor cores
//               (h as a bf16 hi + lo pair, so it keeps ~16 bits) into one of
//               eight TMEM accumulators; completions free the B part of a
//               ring slot;
//   warps 2, 3  operands: per unit, the token list and h of the unit's slice
//               from global memory as bf16 hi / lo operand tiles (128-byte
//               swizzle), double-buffered one unit ahead;
//   warps 4-11  epilogue, two teams of four that take alternate stages: each
//               warp reads its 32 accumulator rows (tcgen05.ld), adds base in
//               fp32 and writes the rounded rows back in place, then stores
//               its 32 x 64 piece with one TMA box store (a full tile of
//               consecutive tokens) or 16-byte row stores through the token
//               list; a slot is handed back once its stores have read it.
// Every wait is bounded; on a timeout the kernel sets a status bit and ends.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kStWarps = 12;
constexpr int kStThreads = kStWarps * 32;
constexpr int kStCols = 64;              // output columns per stage
constexpr int kStAcc = 8;                // TMEM accumulators of kStCols columns (all 512 columns)
constexpr int kStTileBytes = 128 * 128;  // 128 rows x 64 bf16: a base stage or an operand tile
constexpr int kStOpBar = 3;              // named barrier of the operand warps
constexpr int kStEpiWarp0 = 4;

struct StreamParams {
    CUtensorMap tmB[kMaxSlices];  // slice j of B: L * b_rows[j] rows of R bf16, box R x 64
    CUtensorMap tmY;              // base / y (s rows, N): box 64 x 128, 128-byte swizzle (loads)
    CUtensorMap tmYs;             // the same, box 64 x 32 (one epilogue warp's store)
    CUtensorMap tmYg;             // the same, box 64 x 1 (4-row gathers)
    LoraParams p;
    int runcap, max_segments;
    int cb;                       // columns of a unit (multiple of 64)
    int upt;                      // units per tile: sum over slices of ceil(width / cb)
    int S;                        // ring slots
    int o_bar, o_run, o_tok, o_op, o_ring;
    int slot_bytes;               // base tile + B tile
};

}  // namespace csgmv
