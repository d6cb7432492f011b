"""The named workloads at their full sizes, each through the csgmv_qkv path
the benchmark times.  The benchmark passes an h workspace to every
csgmv_qkv call, so the library takes a two-kernel path (a shrink into the
fp32 workspace, then an expand) wherever that is its choice: decode QKV (the
cluster-free decode kernels), prefill gate_up and skewed down_proj (the
streaming tcgen05 shrink and expand on 128-token tiles) and both lm_head
workloads (vocabulary-wide outputs on 16-token tiles: the small-tile shrink
and expand-only launches).  The decode QKV and lm_head decode tests also run
the one-kernel fused path (no workspace).  Each test asserts how many kernels its call
launches, with the same rule the benchmark uses to count them.

Decode and lm_head are compared element by element; the prefill workloads on
sampled token rows (every column of each sampled row), which the oracle
computes one by one."""
import numpy as np
import pytest
import torch

import bench
import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, dev_bf16, dev_f32, dev_i32, f64, host_bits, oracle_fused, run_fused

pytestmark = pytest.mark.gpu


def sample_rows(w, n=192, seed=0):
    starts = np.concatenate([[0], np.cumsum(w.req_lens)])
    rows = set()
    for i in range(w.bs):  # first and last token of every request
        if w.req_lens[i] > 0:
            rows.add(int(starts[i]))
            rows.add(int(starts[i + 1] - 1))
    rng = np.random.default_rng(seed)
    rows.update(int(t) for t in rng.integers(0, w.s, size=n))
    return np.array(sorted(rows))


@pytest.mark.parametrize("workspace", [True, False], ids=["workspace", "on-chip"])
def test_decode_qkv_full(workspace):
    """bs 256 x 1 token on 8 slots: with a workspace (the benchmark's call)
    the decode shrink and expand, without one the fused cluster kernel."""
    w = wl.decode_qkv()
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=workspace)
        if workspace:
            assert bench.qkv_kernels(w, bi) == 2
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"decode qkv base={base} workspace={workspace}")


@pytest.mark.parametrize("workspace", [True, False], ids=["workspace", "on-chip"])
def test_lm_head_decode_full(workspace):
    """bs 512 x 1 token onto 128256 columns: with a workspace (the benchmark's
    call) the shrink writes fp32 h and the expand-only launch spreads column
    blocks over every SM; without one the fused kernel keeps h on chip."""
    w = wl.lm_head_decode()
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=workspace)
        if workspace:
            assert bench.qkv_kernels(w, bi) == 2
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"lm_head decode base={base} workspace={workspace}")


def test_lm_head_pruned_full():
    """The benchmarked pruned lm_head pass: 64 requests with one pruned token
    each on 32 slots of rank 32, batch info from the pruned lm_head builder
    (identity permutation, request order), csgmv_qkv onto 128256 columns
    through a NaN-filled workspace, every output element against the oracle."""
    w = wl.lm_head_pruned()
    assert w.meta["builder"] == "lm_head"
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    lens, ad = dev_i32(w.req_lens), dev_i32(w.req_adapter)
    ranks, scal = dev_i32(w.ranks), dev_f32(w.scalings)
    for base in (True, False):
        bi = B.BatchInfo(w.bs, w.s, w.s + 1, max_loras=w.L, max_rank=w.R)
        B.csgmv_build_lm_head_batch_info(bi, lens, ad, w.s, ranks, scal, max_chunk_size=w.max_chunk_size,
                                         use_cuda_graph=True)
        assert bench.qkv_kernels(w, bi) == 2
        y = dev_bf16(w.base) if base else torch.zeros((w.s, w.N), dtype=torch.bfloat16, device="cuda")
        ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, w.c) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
        B.csgmv_qkv(x, A, Bm, w.offsets, w.c, w.N, y, bi, workspace=ws)
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        ref_bi = oracle.build_lm_head_batch_info(w.req_lens, w.req_adapter, bi.chunk_size)
        n = int(bi.num_segments.item())
        assert n == ref_bi["num_segments"]
        assert np.array_equal(bi.seg_indptr[:n + 1].cpu().numpy(), ref_bi["seg_indptr"])
        assert np.array_equal(bi.weight_indices[:n].cpu().numpy(), ref_bi["weight_indices"])
        assert_close(f64(host_bits(y)), oracle_fused(w, base=base), f"lm_head pruned base={base}")


@pytest.mark.parametrize("workspace", [False, True], ids=["on-chip", "workspace"])
def test_prefill_gate_up_sampled(workspace):
    """Both csgmv_qkv paths at full size: h on chip, and the two-kernel path
    through a workspace that the bench uses."""
    w = wl.prefill_gate_up()
    rows = sample_rows(w)
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=workspace)
        if workspace:
            assert bench.qkv_kernels(w, bi) == 2
        assert bi.device_status() == 0
        assert_close(f64(y[rows]), oracle_fused(w, base=base, rows=rows), f"prefill gate_up base={base}")


def test_skewed_down_proj_chunk_sweep():
    """Chunk sizes 16 / 32 / 64 / 128 through the benchmark's call (with a
    workspace): every result within tolerance of the oracle on sampled rows,
    and all four bit-identical (chunks only group tokens of one slot)."""
    w = wl.skewed_down_proj(chunk=128)
    rows = sample_rows(w)
    ref = oracle_fused(w, rows=rows)
    first = None
    for chunk in (16, 32, 64, 128):
        y, bi = run_fused(w, chunk_override=chunk, workspace=True)
        assert bi.device_status() == 0 and bi.chunk_size == chunk
        assert_close(f64(y[rows]), ref, f"skewed down_proj chunk={chunk}")
        if first is None:
            first = y
        else:
            assert np.array_equal(y, first), "result depends on the chunk size"
