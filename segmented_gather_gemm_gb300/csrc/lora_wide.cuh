// Expand of short slot runs onto a wide output (a vocabulary-wide lm_head:
// sglang chunked_backend.py run_lora_b_sgemm on the pruned lm_head batch,
// _build_lm_head_batch_info; shapes from base_backend.py), reading h from the
// csgmv_qkv workspace.
//
// A tile is up to TM tokens of one slot (any positions); a unit is a tile and
// a block of its output columns; a unit streams its columns in stages of NT
// columns.  Per stage the slot's B rows (NT rows of R, TMA boxes) and the
// tile's base rows (one bulk copy per token) land in a ring slot.  Warps:
//   load     issues a stage's copies as soon as its ring slot is free;
//   consume  sixteen warps, NT / 16 columns each: h as bf16 hi / lo mma.sync
//            fragments (built once per unit), B fragments by ldmatrix, and
//            y = base + sigma h B^T stored straight from registers (a quad
//            of lanes writes 16 consecutive bytes of a row), after which
//            they free the slot.
// No barrier spans the CTA inside the stream: each stage has a full barrier
// (the copies' bytes) and an empty barrier (the consumer warps).  A stage of
// a short tile is little arithmetic but a long chain of dependent
// instructions per warp, so the columns go to many warps.  B for all
// columns of a slot is read once per tile, so tiles of 32 tokens keep the B
// traffic of a slot with up to 32 tokens at one pass.  All waits are
// bounded.
#pragma once

#include "lora_tma.cuh"

namespace csgmv {

constexpr int kWideConsumers = 16;
constexpr int kWideWarps = 2 + kWideConsumers;  // load, one spare, consumers
constexpr int kWideThreads = kWideWarps * 32;

struct WideParams {
    CUtensorMap tmB;               // B (L*N rows, R): box R x 256, swizzle of the R*2-byte row
    CUtensorMap tmBs[kMaxSlices];  // B per slice tensor (p.b_tuple): box R x 64
    LoraParams p;
    int runcap, max_segments;
    int nt;           // columns per stage (256 or 512)
    int cb;           // columns per unit (a multiple of nt)
    int S;            // ring stages
    int ypitch;       // bytes per staged base row (nt * 2 + 16)
    int stage_bytes;  // base rows (tm * ypitch, rounded to 1024) + B rows (nt * R * 2)
    int b_off;        // offset of the B rows in a stage
    int o_bar, o_run, o_ring;
};

}  // namespace csgmv
