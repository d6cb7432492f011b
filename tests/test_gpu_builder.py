"""Device batch builder (csgmv_build_batch_info) against the oracle builder:
bit-exact permutation, segments, padding, slot tables and request fields."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from tests.gpu_helpers import dev_f32, dev_i32

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def gpu_build(lens, adapter, ranks, scal, num_tokens=None, max_chunk=128, override=0, graph=False,
              capacity=None, R=64):
    lens = np.asarray(lens, np.int32)
    adapter = np.asarray(adapter, np.int32)
    s = int(lens.sum()) if num_tokens is None else num_tokens
    L = len(ranks)
    if capacity is None:
        bi = B.BatchInfo.for_batch(len(lens), max(s, int(lens.clip(0).sum())), L, R,
                                   min_chunk=min(16, override) if override else 16)
    else:
        bi = B.BatchInfo(*capacity, max_loras=L, max_rank=R)
    bi.seg_indptr.fill_(-5)
    bi.weight_indices.fill_(-5)
    B.csgmv_build_batch_info(bi, dev_i32(lens), dev_i32(adapter), s, dev_i32(ranks), dev_f32(scal),
                             max_chunk_size=max_chunk, chunk_size_override=override, use_cuda_graph=graph)
    torch.cuda.synchronize()
    return bi


def compare(bi, lens, adapter, chunk, graph=False):
    ref = oracle.build_batch_info(lens, adapter, chunk, use_cuda_graph=graph,
                                  max_segments=bi.c.max_segments if graph else None)
    n = int(bi.num_segments.item())
    s = int(np.sum(lens))
    assert bi.device_status() == 0
    assert int(bi.max_len.item()) == chunk == bi.chunk_size
    assert n == ref["num_segments"]
    assert np.array_equal(bi.permutation[:s].cpu().numpy(), ref["permutation"])
    if graph:
        ms = bi.c.max_segments
        assert np.array_equal(bi.weight_indices[:ms].cpu().numpy(), ref["weight_indices"])
        assert np.array_equal(bi.seg_indptr[:ms + 1].cpu().numpy(), ref["seg_indptr"])
    else:
        assert np.array_equal(bi.weight_indices[:n].cpu().numpy(), ref["weight_indices"])
        assert np.array_equal(bi.seg_indptr[:n + 1].cpu().numpy(), ref["seg_indptr"])
    bs = len(lens)
    assert np.array_equal(bi.req_seg_indptr[:bs + 1].cpu().numpy(), ref["req_seg_indptr"])
    assert np.array_equal(bi.req_weight_indices[:bs].cpu().numpy(), ref["req_weight_indices"])
    want = expected_tiles(ref)
    got = bi.tile_table.cpu().numpy()
    assert int(got[0]) == len(want) and not got[1:4].any()
    assert np.array_equal(got[4:4 + 4 * len(want)].reshape(-1, 4), np.array(want, np.int32).reshape(-1, 4))


def expected_tiles(ref, tm=64):
    """Decode tiles from the oracle's segments: each maximal stretch of
    segments on one slot (a slot run of n tokens) cut into ceil(n / tm)
    tiles of balanced size, records (slot, first position, tokens, 0)."""
    n = ref["num_segments"]
    w, ip = ref["weight_indices"][:n], ref["seg_indptr"][:n + 1]
    tiles, k = [], 0
    while k < n:
        e = k
        while e + 1 < n and w[e + 1] == w[k]:
            e += 1
        p0, cnt = int(ip[k]), int(ip[e + 1] - ip[k])
        nt = -(-cnt // tm)
        for i in range(nt):
            lo, hi = i * cnt // nt, (i + 1) * cnt // nt
            tiles.append((int(w[k]), p0 + lo, hi - lo, 0))
        k = e + 1
    return tiles


def test_tiny_golden():
    g = json.load(open(os.path.join(GOLDEN, "tiny_batch_info.json")))
    bi = gpu_build(g["req_lens"], g["req_adapter"], [8, 8, 0], [2.0, 2.0, 2.0], override=16)
    assert bi.permutation[:64].cpu().tolist() == g["permutation"]
    assert bi.weight_indices[:4].cpu().tolist() == g["weight_indices"]
    assert bi.seg_indptr[:5].cpu().tolist() == g["seg_indptr"]
    assert bi.lora_ranks.cpu().tolist() == [8, 8, 0]
    assert bi.req_seg_indptr.cpu().tolist() == g["req_seg_indptr"]
    gb = gpu_build(g["req_lens"], g["req_adapter"], [8, 8, 0], [2.0] * 3, override=16, graph=True,
                   capacity=(4, 64, g["graph_max_segments"]))
    assert gb.weight_indices.cpu().tolist() == g["graph_weight_indices"]
    assert gb.seg_indptr.cpu().tolist() == g["graph_seg_indptr"]


def test_worked_examples():
    p = json.load(open(os.path.join(GOLDEN, "permutation_worked_example.json")))
    sg = json.load(open(os.path.join(GOLDEN, "segments_worked_example.json")))
    bi = gpu_build(p["extend_seq_lens"], p["seq_weight_indices"], [4, 4], [1.0, 1.0], override=3)
    assert bi.permutation[:6].cpu().tolist() == p["permutation"]
    assert bi.weight_indices[:3].cpu().tolist() == sg["weight_indices"]
    assert bi.seg_indptr[:4].cpu().tolist() == sg["seg_indptr"]


@pytest.mark.parametrize("seed", range(24))
def test_random_batches(seed):
    rng = np.random.default_rng(500 + seed)
    bs = int(rng.integers(1, 80))
    L = int(rng.integers(1, 40))
    lens = rng.integers(0, 300, size=bs) if seed % 3 else np.ones(bs, np.int64)
    lens[rng.random(bs) < 0.1] = 0
    adapter = rng.integers(0, L, size=bs)
    ranks = rng.integers(0, 65, size=L)
    scal = rng.uniform(0, 3, size=L).astype(np.float32)
    s = int(lens.sum())
    override = int(rng.choice([0, 0, 16, 32, 64, 128, 7]))
    max_chunk = int(rng.choice([8, 16, 64, 128, 100]))
    chunk = override if override else oracle.chunk_size(s, max_chunk)
    graph = seed % 2 == 1
    cap = None
    if graph:
        ms, mt = oracle.capacity(bs, int(lens.max()) if bs else 1)
        cap = (bs, mt, ms + (0 if chunk >= 16 else s))
    bi = gpu_build(lens, adapter, ranks, scal, max_chunk=max_chunk, override=override, graph=graph, capacity=cap)
    compare(bi, lens, adapter, chunk, graph=graph)
    assert np.array_equal(bi.lora_ranks.cpu().numpy(), ranks)
    assert np.array_equal(bi.scalings.cpu().numpy(), scal)


def test_many_requests_and_slots():
    # > 1024 requests: several request tiles inside the single-CTA builder
    rng = np.random.default_rng(7)
    bs, L = 3000, 700
    lens = rng.integers(0, 9, size=bs)
    adapter = rng.integers(0, L, size=bs)
    bi = gpu_build(lens, adapter, np.full(L, 16), np.ones(L, np.float32), override=16)
    compare(bi, lens, adapter, 16)


def test_empty_batch():
    bi = gpu_build([], [], [8], [1.0], num_tokens=0)
    assert int(bi.num_segments.item()) == 0 and bi.device_status() == 0


def test_device_errors_leave_zero_segments():
    bi = gpu_build([3, 4], [0, 5], [8, 8], [1.0, 1.0])
    assert bi.device_status() & 1 and int(bi.num_segments.item()) == 0
    bi = gpu_build([3, 4], [0, 1], [8, 8], [1.0, 1.0], num_tokens=6)
    assert bi.device_status() & 32 and int(bi.num_segments.item()) == 0
    bi = gpu_build([3, -1], [0, 1], [8, 8], [1.0, 1.0], num_tokens=2)
    assert bi.device_status() & 32
    bi = gpu_build([3, 4], [0, 1], [8, 80], [1.0, 1.0])
    assert bi.device_status() & 2
    # more segments than the buffers hold
    bi = gpu_build([40, 40], [0, 1], [8, 8], [1.0, 1.0], override=16, graph=True, capacity=(2, 80, 3))
    assert bi.device_status() & 16 and int(bi.num_segments.item()) == 0
    # a good build afterwards resets the status
    bi2 = gpu_build([3, 4], [0, 1], [8, 8], [1.0, 1.0])
    assert bi2.device_status() == 0
