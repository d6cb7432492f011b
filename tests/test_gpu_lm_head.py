"""Pruned lm_head batch info (csgmv_build_lm_head_batch_info) against the
oracle: bit-exact segments, identity permutation and padding, then the LoRA
delta over the pruned rows with that batch info."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, dev_bf16, dev_f32, dev_i32, host_f64

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def lm_build(lens, adapter, ranks, scal, max_chunk=128, graph=False, capacity=None, R=64, override=0):
    lens = np.asarray(lens, np.int32)
    adapter = np.asarray(adapter, np.int32)
    s = int(lens.sum())
    L = len(ranks)
    if capacity is None:  # runs can be as many as requests: room for one segment per token
        bi = B.BatchInfo(len(lens), max(s, 1), max(s, 1) + 1, max_loras=L, max_rank=R)
    else:
        bi = B.BatchInfo(*capacity, max_loras=L, max_rank=R)
    bi.seg_indptr.fill_(-5)
    bi.weight_indices.fill_(-5)
    bi.permutation.fill_(-5)
    B.csgmv_build_lm_head_batch_info(bi, dev_i32(lens), dev_i32(adapter), s, dev_i32(ranks), dev_f32(scal),
                                     max_chunk_size=max_chunk, chunk_size_override=override, use_cuda_graph=graph)
    torch.cuda.synchronize()
    return bi


def lm_compare(bi, lens, adapter, graph=False):
    s = int(np.sum(lens))
    chunk = bi.chunk_size
    ref = oracle.build_lm_head_batch_info(lens, adapter, chunk, use_cuda_graph=graph,
                                          max_segments=bi.c.max_segments if graph else None)
    n = int(bi.num_segments.item())
    assert bi.device_status() == 0
    assert n == ref["num_segments"]
    assert np.array_equal(bi.permutation[:s].cpu().numpy(), ref["permutation"])
    ms = bi.c.max_segments if graph else n
    assert np.array_equal(bi.weight_indices[:ms].cpu().numpy(), ref["weight_indices"])
    assert np.array_equal(bi.seg_indptr[:ms + 1].cpu().numpy(), ref["seg_indptr"])


def test_lm_head_hand_derived():
    with open(os.path.join(GOLDEN, "lm_head_batch_info.json")) as f:
        g = json.load(f)
    L = max(g["req_adapter"]) + 1
    bi = lm_build(g["pruned_lens"], g["req_adapter"], np.full(L, 16), np.ones(L, np.float32),
                  override=g["chunk_size"], graph=True,
                  capacity=(len(g["pruned_lens"]), 11, g["graph_max_segments"]))
    assert bi.device_status() == 0
    assert int(bi.num_segments.item()) == len(g["weight_indices"])
    assert bi.permutation[:11].cpu().tolist() == g["permutation"]
    assert bi.weight_indices[:6].cpu().tolist() == g["graph_weight_indices"]
    assert bi.seg_indptr[:7].cpu().tolist() == g["graph_seg_indptr"]
    assert int(bi.tile_table[0].item()) == -1  # no decode tiles from this builder
    # per-request fields: first pruned token and slot of every request
    starts = np.concatenate([[0], np.cumsum(g["pruned_lens"])])
    assert bi.req_seg_indptr[:len(starts)].cpu().tolist() == starts.tolist()
    assert bi.req_weight_indices[:len(g["req_adapter"])].cpu().tolist() == list(g["req_adapter"])


@pytest.mark.parametrize("seed", range(8))
def test_lm_head_random_batches(seed):
    rng = np.random.default_rng(500 + seed)
    bs = int(rng.integers(1, 1500))
    L = int(rng.integers(1, 40))
    lens = rng.integers(0, 4, size=bs) * (rng.random(bs) < 0.6)
    if seed % 4 == 0:
        lens = rng.integers(0, 40, size=bs)  # long pruned runs: many segments per run, several token tiles
    adapter = rng.integers(0, L, size=bs)
    graph = seed % 2 == 1
    bi = lm_build(lens, adapter, np.full(L, 16), np.ones(L, np.float32), graph=graph,
                  capacity=(bs, max(int(lens.sum()), 1), max(int(lens.sum()), 1) + 8) if graph else None)
    lm_compare(bi, lens, adapter, graph=graph)


def test_lm_head_bad_slot_gives_zero_segments():
    bi = lm_build([2, 3], [0, 5], np.full(2, 16), np.ones(2, np.float32))
    assert bi.device_status() & 1  # BAD_ADAPTER
    assert int(bi.num_segments.item()) == 0


def test_lm_head_delta_over_pruned_rows():
    """The pruned rows of an lm_head-shaped projection (one to three rows per
    request, in request order) through csgmv_qkv with the lm_head batch info."""
    rng = np.random.default_rng(9)
    bs, L, R, K, N = 300, 12, 32, 512, 2048
    lens = rng.integers(0, 4, size=bs).astype(np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    w = wl.random_lora(17, bs=4, max_len=8, K=K, N_slices=[N], R=R, L=L)  # slot weights, ranks, scalings
    ranks, scal = w.ranks, w.scalings
    s = int(lens.sum())
    x = wl.normal_bf16(rng, (s, K), 0.5)
    base = wl.normal_bf16(rng, (s, N), 0.5)
    bi = lm_build(lens, adapter, ranks, scal, R=R)
    assert bi.device_status() == 0
    y = dev_bf16(base)
    B.csgmv_qkv(dev_bf16(x), dev_bf16(w.A), dev_bf16(w.B), [0, N], 1, N, y, bi)
    torch.cuda.synchronize()
    assert bi.device_status() == 0
    ta = np.repeat(adapter, lens).astype(np.int32)
    ref = oracle.fused(x, w.A, w.B, [0, N], 1, ta, ranks, scal, base)
    assert_close(host_f64(y), ref, "lm_head pruned rows")


def test_lm_head_vocabulary_wide_grouped_tiles():
    """The pruned rows of a vocabulary-wide lm_head through csgmv_qkv with a
    workspace: the expand groups each slot's tokens from segments spread over
    the whole batch (request order), some slots holding more than one 16-token
    tile; every output row against the oracle, and rows of zero-length
    requests absent."""
    rng = np.random.default_rng(23)
    bs, L, R, K, N = 200, 32, 32, 256, 33024
    lens = rng.integers(0, 4, size=bs).astype(np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    adapter[:40] = 3  # one slot with well over 16 tokens in many segments
    w = wl.random_lora(29, bs=4, max_len=8, K=K, N_slices=[N], R=R, L=L)
    ranks, scal = w.ranks, w.scalings
    s = int(lens.sum())
    x = wl.normal_bf16(rng, (s, K), 0.5)
    base = wl.normal_bf16(rng, (s, N), 0.5)
    bi = lm_build(lens, adapter, ranks, scal, R=R)
    assert bi.device_status() == 0
    ws = torch.empty(B.csgmv_qkv_workspace_bytes(bi, 1) // 4, dtype=torch.float32, device="cuda")
    assert B.csgmv_qkv_path(bi, K, N, [0, N], 1, ws.numel() * 4) == "small_split"
    y = dev_bf16(base)
    B.csgmv_qkv(dev_bf16(x), dev_bf16(w.A), dev_bf16(w.B), [0, N], 1, N, y, bi, workspace=ws)
    torch.cuda.synchronize()
    assert bi.device_status() == 0
    ta = np.repeat(adapter, lens).astype(np.int32)
    assert np.sum(ta == 3) > 32
    ref = oracle.fused(x, w.A, w.B, [0, N], 1, ta, ranks, scal, base)
    assert_close(host_f64(y), ref, "vocabulary-wide lm_head rows")
