// Expand of short slot runs onto a wide output (a vocabulary-wide lm_head:
// sglang chunked_backend.py run_lora_b_sgemm on the pruned lm_head batch,
// _build_lm_head_batch_info; shapes from base_backend.py), reading h from the
// csgmv_qkv workspace.
//
// A tile is up to TM = 16 tokens of one slot (any positions); a unit is a
// tile and a block of its output columns; a unit streams its columns in
// stages of NT columns.  Per stage the slot's B rows (NT rows of R, TMA
// boxes) and the tile's base rows (one bulk copy per token) land in a ring
// slot.  Warps:
//   load     issues a stage's copies as soon as its ring slot is free;
//   h        (one output slice) the spare warp builds each unit's tokens and
//            h as bf16 hi / lo mma.sync fragments into one of two shared
//            buffers, a unit ahead of the consumers, so that a unit starts
//            without a round of global loads;
//   consume  sixteen warps, NT / 16 columns each: the unit's h fragments
//            (from the spare warp, or loaded per slice), B fragments by
//            ldmatrix, and y = base + sigma h B^T stored straight from
//            registers (16 consecutive bytes of a row per lane), after which
//            they free the slot.
// Tiles group a slot's tokens wherever its segments lie (a pruned lm_head
// batch keeps its requests in request order, so one slot's tokens are spread
// over several segments): every token of slot w goes to w's tiles, so B rows
// of a slot are read once per TM of its tokens.  Rows of a tile need no
// order, since every output row depends on its own h row alone.
// No barrier spans the CTA inside the stream: each stage has a full barrier
// (the copies' bytes) and an empty barrier (the consumer warps).  A stage of
// a short tile is little arithmetic but a long chain of dependent
// instructions per warp, so the columns go to many warps.  All waits are
// bounded.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kWideConsumers = 16;
constexpr int kWideGroupBytes = 32 * 1024;  // shared memory a grouped tile table may take

// Ints of a grouped tile table (lora_wide.cu wide_group).
inline size_t wide_group_ints(int nslot, int segcap, int tokcap) {
    return (size_t)5 * nslot + 3 + 4 * (size_t)segcap + tokcap + 32;
}
constexpr int kWideWarps = 2 + kWideConsumers;  // load, h, consumers
constexpr int kWideHfInts = 4 * 2 * 4 * 32;      // h fragments of one 16-token unit: k16 steps x hi/lo x regs x lanes
constexpr int kWideThreads = kWideWarps * 32;

struct WideParams {
    CUtensorMap tmB;               // B (L*N rows, R): box R x 256, swizzle of the R*2-byte row
    CUtensorMap tmBs[kMaxSlices];  // B per slice tensor (p.b_tuple): box R x 64
    LoraParams p;
    int runcap, max_segments;
    int grouped;      // tiles by slot (nslot, segcap, tokcap below); else tiles of segment runs
    int nslot;        // slots the grouped table counts (max_loras)
    int segcap;       // segments it holds (max_segments)
    int tokcap;       // positions it holds (num_tokens)
    int nt;           // columns per stage (256 or 512)
    int cb;           // columns per unit (a multiple of nt)
    int S;            // ring stages
    int ypitch;       // bytes per staged base row (nt * 2 + 16)
    int stage_bytes;  // base rows (tm * ypitch, rounded to 1024) + B rows (nt * R * 2)
    int b_off;        // offset of the B rows in a stage
    int o_bar, o_hbar, o_run, o_hf, o_ring;  // o_hbar: hfull[2], hempty[2]; o_hf: fragments[2], tokens[2][32]
};

}  // namespace csgmv
