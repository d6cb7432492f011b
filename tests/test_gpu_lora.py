"""Shrink, expand and fused shrink->expand kernels against the fp64 oracle on
seeded inputs: several token tiles with ragged tails, odd ranks, rank-0 slots,
one to three slices, poison in every padding row/column, CUDA-graph replay of
a different batch, chunk-size invariance."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import (assert_close, build_batch, dev_bf16, dev_f32, dev_i32, f64, host_bits,
                               host_f64, oracle_fused, run_fused)

pytestmark = pytest.mark.gpu

# (seed, bs, max_len, K, slices, R, L) -- small s runs the decode tiles, the
# large-s cases (s > 1024 on few slots) run the 128- / 64-token prefill tiles.
CASES = [
    (1, 6, 9, 64, [32], 8, 3),
    (2, 20, 1, 520, [64, 16, 16], 16, 5),
    (3, 9, 40, 136, [128, 64], 32, 4),
    (4, 3, 600, 256, [96], 64, 2),
    (5, 4, 500, 264, [64, 64, 32], 64, 3),
    (6, 5, 450, 128, [40, 24], 32, 2),
    (7, 64, 1, 4096, [256, 64, 64], 16, 8),
    (8, 2, 900, 72, [16], 8, 1),
    # output columns well above K
    (9, 3, 700, 128, [256, 128], 64, 3),
    (10, 4, 500, 64, [128, 64, 64], 32, 3),
    (11, 3, 400, 96, [160], 16, 2),
]


def make(seed, bs, max_len, K, slices, R, L, pad=None, min_len=0):
    return wl.random_lora(seed, bs=bs, max_len=max_len, K=K, N_slices=slices, R=R, L=L,
                          rank_choices=list(range(1, R + 1)), zero_rank_prob=0.2, std=0.5,
                          pad_value=pad, min_len=min_len)


@pytest.mark.parametrize("case", CASES, ids=[f"case{c[0]}" for c in CASES])
def test_fused_matches_oracle(case):
    w = make(*case, min_len=1 if case[2] == 1 else 0)
    for base in (True, False):
        y, bi = run_fused(w, base=base)
        assert bi.device_status() == 0
        ref = oracle_fused(w, base=base)
        assert_close(f64(y), ref, f"fused base={base} {case}")


@pytest.mark.parametrize("case", [CASES[3], CASES[4], CASES[8], CASES[9]], ids=["c1r64", "c3r64", "c2r64", "c3r32"])
def test_fused_with_workspace_matches_oracle(case):
    """csgmv_qkv with a workspace (two-kernel path for long slot runs) gives
    the oracle's result, with and without base."""
    w = make(*case)
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=True)
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"fused+workspace base={base} {case}")
    # NaN in every padding row of A and column of B changes nothing
    y0, _ = run_fused(w, workspace=True)
    y1, _ = run_fused(make(*case, pad=float("nan")), workspace=True)
    assert np.array_equal(y0, y1), f"padding leaked into the output ({case})"


# (seed, bs, max_len, K, slices, R, L): short requests on a handful of slots and
# at least 32768 output columns, so that csgmv_qkv with a workspace runs the
# 16-token shrink into the workspace and then the expand-only launch
# (at most 16 tokens a slot on average: the wide kernel; more: the small-tile
# kernel's expand-only launch)
WIDE = [
    (12, 40, 1, 256, [33024], 32, 6),
    (13, 24, 3, 136, [16384, 16400], 8, 5),
    (14, 30, 2, 128, [16384, 8192, 8256], 64, 8),
    (16, 40, 4, 128, [33024], 16, 3),  # about 30 tokens a slot: the small-tile expand
]


@pytest.mark.parametrize("case", WIDE, ids=["c1r32", "c2r8", "c3r64", "c1r16-small"])
def test_wide_output_split_matches_oracle(case):
    """Vocabulary-wide outputs on small tiles take the two-kernel path: the
    oracle's result, with and without base, and bit-identical output with NaN
    in every padding row and column."""
    w = make(*case, min_len=1)
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=True)
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"wide split base={base} {case}")
    y0, _ = run_fused(w, workspace=True)
    y1, _ = run_fused(make(*case, pad=float("nan"), min_len=1), workspace=True)
    assert np.array_equal(y0, y1), f"padding leaked into the output ({case})"


@pytest.mark.parametrize("h_f32", [True, False])
@pytest.mark.parametrize("slices", [[33024], [16392, 16392]], ids=["one-slice", "slice-edge-mid-pair"])
def test_wide_expand_only(slices, h_f32):
    """csgmv_expand onto a vocabulary-wide output with short slot runs (the
    wide kernel): accumulate on and off (rank-0 slots then write zeros),
    ragged ranks, fp32 and bf16 h, and a slice edge inside a 16-column pair."""
    w = make(15, 40, 1, 64, slices, 32, 6, min_len=1)
    bi = build_batch(w)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    cR = w.c * w.R
    h = torch.zeros((w.s, cR), dtype=torch.float32 if h_f32 else torch.bfloat16, device="cuda")
    B.csgmv_shrink(x, A, w.c, h, bi)
    torch.cuda.synchronize()
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    hg = host_f64(h)
    widest = int(np.max(np.diff(w.offsets)))
    for acc in (True, False):
        out = dev_bf16(w.base) if acc else torch.full((w.s, w.N), 3.0, dtype=torch.bfloat16, device="cuda")
        B.csgmv_expand(h, Bm, w.offsets, w.c, widest, out, acc, bi)
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        yref = oracle.expand(hg, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base if acc else None)
        assert_close(f64(host_bits(out)), yref, f"wide expand accumulate={acc}")


def test_tiny_single_slice_workload():
    w = wl.tiny_single_slice()
    for base in (True, False):
        y, bi = run_fused(w, base=base)
        assert_close(f64(y), oracle_fused(w, base=base), "tiny")
    # slot 2 has rank 0: its request's rows keep base exactly
    y, _ = run_fused(w, base=True)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    assert np.array_equal(y[ta == 2], w.base[ta == 2])


@pytest.mark.parametrize("pad", [1.0e30, float("nan")])
def test_padding_never_read(pad):
    for case in (CASES[2], CASES[4], CASES[6]):
        clean = make(*case)
        dirty = make(*case, pad=pad)
        y0, _ = run_fused(clean)
        y1, _ = run_fused(dirty)
        assert np.array_equal(y0, y1), f"padding leaked into the output ({case})"


@pytest.mark.parametrize("h_f32", [True, False])
@pytest.mark.parametrize("case", [CASES[1], CASES[3], CASES[4]], ids=["c3r16", "c1r64", "c3r64"])
def test_shrink_then_expand(case, h_f32):
    w = make(*case)
    bi = build_batch(w)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    cR = w.c * w.R
    ldh = cR + 8
    h = torch.full((w.s, ldh), 7.0, dtype=torch.float32 if h_f32 else torch.bfloat16, device="cuda")
    B.csgmv_shrink(x, A, w.c, h, bi)
    torch.cuda.synchronize()
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    href = oracle.shrink(w.x, w.A, w.c, ta, w.ranks)
    hg = host_f64(h)
    assert_close(hg[:, :cR], href, "shrink h")
    assert np.all(hg[:, cR:] == 7.0), "shrink wrote beyond c*R"
    for t in range(w.s):
        r = int(w.ranks[ta[t]])
        assert np.all(hg[t, w.c * r:cR] == 0.0)
    widest = int(np.max(np.diff(w.offsets)))
    for acc in (True, False):
        out = dev_bf16(w.base) if acc else torch.full((w.s, w.N), 3.0, dtype=torch.bfloat16, device="cuda")
        B.csgmv_expand(h, Bm, w.offsets, w.c, widest, out, acc, bi)
        torch.cuda.synchronize()
        yref = oracle.expand(hg[:, :cR], w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base if acc else None)
        assert_close(f64(host_bits(out)), yref, f"expand accumulate={acc}")


def test_graph_replay_with_another_batch():
    """Capture build + fused once; replay after writing a different batch
    (other slot assignment, fewer segments) into the same input buffers."""
    bs, L, R, K = 48, 6, 16, 256
    slices = [64, 32, 32]
    wa = wl.random_lora(21, bs=bs, max_len=1, K=K, N_slices=slices, R=R, L=L, zero_rank_prob=0.0, min_len=1)
    wb = wl.random_lora(22, bs=bs, max_len=1, K=K, N_slices=slices, R=R, L=L, zero_rank_prob=0.0, min_len=1)
    wb.req_adapter[:] = np.where(wb.req_adapter % 2 == 0, 1, 4)  # two slots only
    bi = B.BatchInfo.for_cuda_graph(bs, 1, L, R)
    lens, ad = dev_i32(wa.req_lens), dev_i32(wa.req_adapter)
    ranks, scal = dev_i32(wa.ranks), dev_f32(wa.scalings)
    x, A, Bm, y = dev_bf16(wa.x), dev_bf16(wa.A), dev_bf16(wa.B), dev_bf16(wa.base)
    widest = 64
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):  # warm-up outside capture (occupancy queries, attributes)
            B.csgmv_build_batch_info(bi, lens, ad, bs, ranks, scal, use_cuda_graph=True)
            B.csgmv_qkv(x, A, Bm, wa.offsets, 3, widest, y, bi)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.csgmv_build_batch_info(bi, lens, ad, bs, ranks, scal, use_cuda_graph=True)
        B.csgmv_qkv(x, A, Bm, wa.offsets, 3, widest, y, bi)
    for w in (wa, wb, wa):
        nseg = oracle.build_batch_info(w.req_lens, w.req_adapter, oracle.chunk_size(bs, 128))["num_segments"]
        lens.copy_(dev_i32(w.req_lens)); ad.copy_(dev_i32(w.req_adapter))
        ranks.copy_(dev_i32(w.ranks)); scal.copy_(dev_f32(w.scalings))
        x.copy_(dev_bf16(w.x)); A.copy_(dev_bf16(w.A)); Bm.copy_(dev_bf16(w.B)); y.copy_(dev_bf16(w.base))
        g.replay()
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        assert_close(f64(host_bits(y)), oracle_fused(w), "graph replay")
        assert int(bi.num_segments.item()) == nseg


def test_chunk_size_invariance_bit_exact():
    w = make(31, 6, 400, 192, [64, 64], 32, 4, min_len=100)
    outs = []
    for chunk in (16, 32, 64, 128):
        y, _ = run_fused(w, chunk_override=chunk)
        outs.append(y)
    for y in outs[1:]:
        assert np.array_equal(y, outs[0])
    assert_close(f64(outs[0]), oracle_fused(w), "chunk sweep")


def test_single_token_and_empty():
    w = make(41, 1, 1, 64, [16], 8, 1, min_len=1)
    w.ranks[:] = 8
    y, _ = run_fused(w)
    assert_close(f64(y), oracle_fused(w), "s=1")
    e = make(42, 3, 0, 64, [16], 8, 2)
    assert e.s == 0
    bi = build_batch(e)
    out = torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda")
    B.csgmv_qkv(torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"), dev_bf16(e.A), dev_bf16(e.B),
                e.offsets, 1, 16, out, bi)
    torch.cuda.synchronize()


def test_request_order_invariance():
    w = make(51, 12, 60, 128, [32, 32], 16, 4)
    y, _ = run_fused(w)
    order = np.random.default_rng(5).permutation(w.bs)
    starts = np.concatenate([[0], np.cumsum(w.req_lens)])
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in order]).astype(int)
    w2 = make(51, 12, 60, 128, [32, 32], 16, 4)
    w2.req_lens, w2.req_adapter = w.req_lens[order], w.req_adapter[order]
    w2.x, w2.base = w.x[rows], w.base[rows]
    y2, _ = run_fused(w2)
    assert np.array_equal(y2, y[rows])
