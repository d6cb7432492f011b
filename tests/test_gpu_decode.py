"""The decode kernels of csgmv_qkv (a split-K shrink into fp32 planes of the
workspace, then an expand that sums them) against the fp64 oracle: decode
shapes with one to three slices, buffer ranks 8 to 64, ragged and zero slot
ranks, K not a multiple of 64, slot runs longer than one 64-token tile, a
workspace with room for one plane only (the shrink then stages K in several
passes), NaN in the workspace and in every padding row / column, repeated
calls and chunk sizes that must give identical bits, CUDA-graph replay of
another batch, and a bad slot rank."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import (assert_close, build_batch, dev_bf16, dev_f32, dev_i32, f64, host_bits,
                               oracle_fused)

pytestmark = pytest.mark.gpu

# (seed, bs, max_len, K, slices, R, L): mean tokens per slot run at most 48
CASES = [
    (61, 40, 1, 64, [32], 8, 3),
    (62, 20, 3, 520, [64, 16, 16], 16, 5),
    (63, 9, 12, 136, [128, 64], 32, 4),
    (64, 30, 4, 256, [96], 64, 2),
    (65, 64, 1, 4096, [256, 64, 64], 16, 8),
    (66, 200, 1, 1024, [512, 128, 128], 64, 6),
    (67, 12, 90, 192, [64], 16, 12),       # runs of up to ~180 tokens: several tiles per run
    (68, 300, 1, 72, [4096, 1024, 1024], 16, 16),
]


def make(seed, bs, max_len, K, slices, R, L, pad=None, min_len=1):
    return wl.random_lora(seed, bs=bs, max_len=max_len, K=K, N_slices=slices, R=R, L=L,
                          rank_choices=list(range(1, R + 1)), zero_rank_prob=0.2, std=0.5,
                          pad_value=pad, min_len=min_len)


def run(w, base=True, chunk_override=None, ws_floats=None, fill=float("nan")):
    """csgmv_qkv with a workspace (NaN-filled: the result must not depend on
    its contents); ws_floats overrides its size."""
    bi = build_batch(w, chunk_override)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    y = dev_bf16(w.base) if base else torch.zeros((w.s, w.N), dtype=torch.bfloat16, device="cuda")
    n = B.csgmv_qkv_workspace_bytes(bi, w.c) // 4 if ws_floats is None else ws_floats
    ws = torch.full((n,), fill, dtype=torch.float32, device="cuda")
    widest = int(np.max(np.diff(w.offsets)))
    assert B.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, 4 * n) == "decode"
    B.csgmv_qkv(x, A, Bm, w.offsets, w.c, widest, y, bi, workspace=ws)
    torch.cuda.synchronize()
    return host_bits(y), bi


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_decode_path_matches_oracle(case):
    w = make(*case)
    for base in (True, False):
        y, bi = run(w, base=base)
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"decode base={base} {case}")


@pytest.mark.parametrize("case", [CASES[1], CASES[3], CASES[5]], ids=["c3r16", "c1r64", "c3r64"])
def test_padding_and_workspace_contents_never_read(case):
    """NaN in every padding row of A and column of B, and a workspace holding
    zeros instead of NaN, give the same bits."""
    y0, _ = run(make(*case))
    y1, _ = run(make(*case, pad=float("nan")))
    y2, _ = run(make(*case), fill=0.0)
    assert np.array_equal(y0, y1), f"padding leaked into the output ({case})"
    assert np.array_equal(y0, y2), f"workspace contents leaked into the output ({case})"


def test_repeat_and_chunk_size_bit_exact():
    """The planes are summed in part order: repeated calls and every chunk
    size (the same slot runs, so the same tiles and parts) agree bit for bit."""
    w = make(71, 96, 3, 1024, [128, 64, 64], 32, 6)
    outs = [run(w, chunk_override=c)[0] for c in (16, 16, 32, 64, 128)]
    for y in outs[1:]:
        assert np.array_equal(y, outs[0])
    assert_close(f64(outs[0]), oracle_fused(w), "chunk sweep")


def test_one_plane_workspace():
    """Room for a single plane: one part of K per tile, staged in several
    passes of the shrink's K chunks (K = 4096 is 64 chunks)."""
    w = make(72, 64, 1, 4096, [256, 64, 64], 16, 8)
    one = (256 + w.s * w.c * w.R * 4) // 4
    y1, bi = run(w, ws_floats=one)
    assert bi.device_status() == 0
    assert_close(f64(y1), oracle_fused(w), "one plane")
    y2, _ = run(w, ws_floats=2 * one)
    assert_close(f64(y2), oracle_fused(w), "two planes")


def test_single_token_single_slot():
    w = make(73, 1, 1, 64, [16], 8, 1)
    w.ranks[:] = 5
    y, bi = run(w)
    assert bi.device_status() == 0
    assert_close(f64(y), oracle_fused(w), "s=1")


def test_graph_replay_with_another_batch():
    """Build + csgmv_qkv (decode kernels) captured once; replayed after
    writing a different batch into the same buffers."""
    bs, L, R, K = 64, 6, 16, 512
    slices = [128, 64, 64]
    wa = wl.random_lora(74, bs=bs, max_len=1, K=K, N_slices=slices, R=R, L=L, zero_rank_prob=0.0, min_len=1)
    wb = wl.random_lora(75, bs=bs, max_len=1, K=K, N_slices=slices, R=R, L=L, zero_rank_prob=0.0, min_len=1)
    wb.req_adapter[:] = np.where(wb.req_adapter % 2 == 0, 1, 4)
    bi = B.BatchInfo.for_cuda_graph(bs, 1, L, R)
    lens, ad = dev_i32(wa.req_lens), dev_i32(wa.req_adapter)
    ranks, scal = dev_i32(wa.ranks), dev_f32(wa.scalings)
    x, A, Bm, y = dev_bf16(wa.x), dev_bf16(wa.A), dev_bf16(wa.B), dev_bf16(wa.base)
    ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, 3) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):
            B.csgmv_build_batch_info(bi, lens, ad, bs, ranks, scal, use_cuda_graph=True)
            B.csgmv_qkv(x, A, Bm, wa.offsets, 3, 128, y, bi, workspace=ws)
    torch.cuda.synchronize()
    assert B.csgmv_qkv_path(bi, K, wa.N, wa.offsets, 3, 4 * ws.numel()) == "decode"
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.csgmv_build_batch_info(bi, lens, ad, bs, ranks, scal, use_cuda_graph=True)
        B.csgmv_qkv(x, A, Bm, wa.offsets, 3, 128, y, bi, workspace=ws)
    for w in (wa, wb, wa):
        lens.copy_(dev_i32(w.req_lens)); ad.copy_(dev_i32(w.req_adapter))
        ranks.copy_(dev_i32(w.ranks)); scal.copy_(dev_f32(w.scalings))
        x.copy_(dev_bf16(w.x)); A.copy_(dev_bf16(w.A)); Bm.copy_(dev_bf16(w.B)); y.copy_(dev_bf16(w.base))
        g.replay()
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        assert_close(f64(host_bits(y)), oracle_fused(w), "graph replay")


def test_bad_rank_flagged_and_rows_kept():
    """A slot rank above max_rank written into the batch info after the build:
    status bit 2, and that slot's rows keep their base values."""
    w = make(76, 48, 1, 256, [64, 32], 16, 4)
    w.ranks[:] = [16, 9, 12, 4]
    bi = build_batch(w)
    bi.lora_ranks[2] = 17
    x, A, Bm, y = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B), dev_bf16(w.base)
    ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, w.c) // 4,), float("nan"), dtype=torch.float32, device="cuda")
    assert B.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, 4 * ws.numel()) == "decode"
    B.csgmv_qkv(x, A, Bm, w.offsets, w.c, 64, y, bi, workspace=ws)
    torch.cuda.synchronize()
    assert bi.device_status() & 2
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    got = host_bits(y)
    keep = ta == 2
    assert np.array_equal(got[keep], w.base[keep])
    ref = oracle_fused(w)
    assert_close(f64(got[~keep]), ref[~keep], "other slots")


def test_tiles_without_the_builders_table():
    """The kernels' own tiles from the segments (a batch info without a tile
    table, or one the table says was not built) give the same bits as the
    builder's table."""
    w = make(78, 70, 3, 512, [128, 64, 64], 16, 9)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    lens, ad = dev_i32(w.req_lens), dev_i32(w.req_adapter)
    ranks, scal = dev_i32(w.ranks), dev_f32(w.scalings)
    outs = []
    for mode in ("table", "no_table", "not_built"):
        bi = B.BatchInfo.for_batch(w.bs, w.s, w.L, w.R, with_tile_table=mode != "no_table")
        B.csgmv_build_batch_info(bi, lens, ad, w.s, ranks, scal, max_chunk_size=w.max_chunk_size)
        if mode == "not_built":
            bi.tile_table[0] = -1
        y = dev_bf16(w.base)
        ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, w.c) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
        assert B.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, 4 * ws.numel()) == "decode"
        B.csgmv_qkv(x, A, Bm, w.offsets, w.c, 128, y, bi, workspace=ws)
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        outs.append(host_bits(y))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    assert_close(f64(outs[0]), oracle_fused(w), "builder tiles")
