"""Pins of the CPU oracle against things other than itself (CPU only).

Each check ties the oracle to a fact the pages or the mathematics fix: the
worked examples printed in sglang's chunked_backend.py docstrings, the
chunk-size rule, the CUDA-graph capacity and padding rule, brute force written
a different way (Python's stable ``sorted``, a token-walking segmenter, numpy
dense per-token weight deltas), closed forms (one adapter == dense matmul) and
invariants (rank 0 leaves base unchanged, request-order invariance, linearity
in the scaling, column indexing for the embedding).
"""
import json
import os

import numpy as np
import pytest

import oracle
from segmented_gather_gemm_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# batch info
# --------------------------------------------------------------------------

def test_chunk_size_rule_table():
    g = golden("chunk_size_rule.json")
    for n, mx, want in g["rows"]:
        assert oracle.chunk_size(n, mx) == want, (n, mx)


def test_graph_capacity_table():
    g = golden("graph_capacity.json")
    for bs, ntpb, ms, mt in g["rows"]:
        assert oracle.capacity(bs, ntpb) == (ms, mt)


def test_permutation_worked_example():
    g = golden("permutation_worked_example.json")
    ta = oracle.token_adapter(g["extend_seq_lens"], g["seq_weight_indices"])
    assert ta.tolist() == g["row_weight_indices"]
    bi = oracle.build_batch_info(g["extend_seq_lens"], g["seq_weight_indices"], chunk=16)
    assert bi["permutation"].tolist() == g["permutation"]
    assert bi["weights_reordered"].tolist() == g["weights_reordered"]


def test_segments_worked_example():
    g = golden("segments_worked_example.json")
    # the docstring's reordered keys are exactly those of the permutation example
    p = golden("permutation_worked_example.json")
    bi = oracle.build_batch_info(p["extend_seq_lens"], p["seq_weight_indices"], chunk=g["chunk_size"])
    assert bi["weights_reordered"].tolist() == g["weights_reordered"]
    assert bi["weight_indices"].tolist() == g["weight_indices"]
    assert bi["seg_indptr"].tolist() == g["seg_indptr"]


def test_tiny_batch_info_hand_derived():
    g = golden("tiny_batch_info.json")
    bi = oracle.build_batch_info(g["req_lens"], g["req_adapter"], chunk=g["chunk_size"])
    assert bi["permutation"].tolist() == g["permutation"]
    assert bi["weight_indices"].tolist() == g["weight_indices"]
    assert bi["seg_indptr"].tolist() == g["seg_indptr"]
    assert bi["req_seg_indptr"].tolist() == g["req_seg_indptr"]
    assert bi["req_weight_indices"].tolist() == g["req_weight_indices"]
    gb = oracle.build_batch_info(g["req_lens"], g["req_adapter"], chunk=g["chunk_size"],
                                 use_cuda_graph=True, max_segments=g["graph_max_segments"])
    assert gb["num_segments"] == 4
    assert gb["weight_indices"].tolist() == g["graph_weight_indices"]
    assert gb["seg_indptr"].tolist() == g["graph_seg_indptr"]


def _brute_batch_info(lens, adapter, chunk):
    """Stable sort with Python's sorted(), then segments by walking tokens."""
    key = []
    for n, a in zip(lens, adapter):
        key += [int(a)] * int(n)
    perm = sorted(range(len(key)), key=lambda t: key[t])
    wi, indptr = [], [0]
    run_key, run_len = None, 0
    for p, t in enumerate(perm):
        k = key[t]
        if k != run_key or run_len == chunk:
            if run_key is not None:
                indptr.append(p)
            wi.append(k)
            run_key, run_len = k, 0
        run_len += 1
    if run_key is not None:
        indptr.append(len(perm))
    return perm, wi, indptr


@pytest.mark.parametrize("seed", range(40))
def test_builder_brute_force(seed):
    rng = np.random.default_rng(1000 + seed)
    bs = int(rng.integers(0, 12))
    L = int(rng.integers(1, 6))
    lens = rng.integers(0, 40, size=bs)
    adapter = rng.integers(0, L, size=bs)
    chunk = int(rng.choice([1, 2, 3, 5, 16, 32, 128]))
    bi = oracle.build_batch_info(lens, adapter, chunk=chunk)
    perm, wi, indptr = _brute_batch_info(lens, adapter, chunk)
    assert bi["permutation"].tolist() == perm
    assert bi["weight_indices"].tolist() == wi
    assert bi["seg_indptr"].tolist() == indptr
    assert bi["num_segments"] == len(wi)


@pytest.mark.parametrize("seed", range(20))
def test_builder_invariants(seed):
    rng = np.random.default_rng(2000 + seed)
    bs = int(rng.integers(1, 64))
    ntpb = int(rng.integers(1, 300))
    L = int(rng.integers(1, 20))
    lens = rng.integers(0, ntpb + 1, size=bs)
    adapter = rng.integers(0, L, size=bs)
    s = int(lens.sum())
    chunk = oracle.chunk_size(s, int(rng.choice([8, 16, 32, 64, 128, 100])))
    max_seg, max_tok = oracle.capacity(bs, ntpb)
    bi = oracle.build_batch_info(lens, adapter, chunk=chunk, use_cuda_graph=True, max_segments=max_seg)
    assert bi["rc"] == 0 and s <= max_tok
    n = bi["num_segments"]
    perm = bi["permutation"]
    assert sorted(perm.tolist()) == list(range(s))  # bijection
    key = oracle.token_adapter(lens, adapter)
    indptr = bi["seg_indptr"]
    assert indptr[0] == 0 and indptr[n] == s
    assert np.all(indptr[n:] == s) and np.all(bi["weight_indices"][n:] == 0)
    for k in range(n):
        seg = perm[indptr[k]:indptr[k + 1]]
        assert 1 <= len(seg) <= chunk
        assert np.all(key[seg] == bi["weight_indices"][k])
        assert np.all(np.diff(seg) > 0)  # stable: original order inside a segment
    counts = np.bincount(key, minlength=L) if s else np.zeros(L, int)
    expect_nseg = sum((int(c) + chunk - 1) // chunk for c in counts)
    assert n == expect_nseg <= max_seg
    for a in range(L):
        got = sum(indptr[k + 1] - indptr[k] for k in range(n) if bi["weight_indices"][k] == a)
        assert got == counts[a]


def test_lm_head_batch_info_hand_derived():
    g = golden("lm_head_batch_info.json")
    bi = oracle.build_lm_head_batch_info(g["pruned_lens"], g["req_adapter"], chunk=g["chunk_size"])
    assert bi["rc"] == 0
    assert bi["permutation"].tolist() == g["permutation"]
    assert bi["weight_indices"].tolist() == g["weight_indices"]
    assert bi["seg_indptr"].tolist() == g["seg_indptr"]
    gb = oracle.build_lm_head_batch_info(g["pruned_lens"], g["req_adapter"], chunk=g["chunk_size"],
                                         use_cuda_graph=True, max_segments=g["graph_max_segments"])
    assert gb["weight_indices"].tolist() == g["graph_weight_indices"]
    assert gb["seg_indptr"].tolist() == g["graph_seg_indptr"]


@pytest.mark.parametrize("seed", range(30))
def test_lm_head_batch_info_invariants(seed):
    """Segments of a pruned lm_head batch, checked token by token: they tile
    [0, s) in order, each holds tokens of one slot only and at most `chunk` of
    them, and a segment ends early only where the slot changes (maximal runs,
    empty requests ignored)."""
    rng = np.random.default_rng(3000 + seed)
    bs = int(rng.integers(1, 80))
    L = int(rng.integers(1, 6))
    lens = rng.integers(0, 6, size=bs) * (rng.random(bs) < 0.7)
    adapter = rng.integers(0, L, size=bs)
    s = int(lens.sum())
    chunk = int(rng.choice([1, 2, 3, 4, 16]))
    bi = oracle.build_lm_head_batch_info(lens, adapter, chunk=chunk)
    assert bi["rc"] == 0
    assert bi["permutation"].tolist() == list(range(s))
    key = np.repeat(adapter, lens)  # slot of every pruned token, in order
    n, indptr, wi = bi["num_segments"], bi["seg_indptr"], bi["weight_indices"]
    assert indptr[0] == 0 and indptr[n] == s
    for k in range(n):
        a, b = indptr[k], indptr[k + 1]
        assert 1 <= b - a <= chunk
        assert np.all(key[a:b] == wi[k])
        if k + 1 < n and wi[k + 1] == wi[k]:
            assert b - a == chunk  # same slot continues: this piece is full
        if k + 1 < n and wi[k + 1] != wi[k]:
            assert key[b] != key[b - 1]


def test_builder_capacity_overflow_reports():
    bi = oracle.build_batch_info([40, 40], [0, 1], chunk=16, use_cuda_graph=True, max_segments=3)
    assert bi["rc"] == -1 and bi["num_segments"] == 0


def test_builder_empty_batch():
    bi = oracle.build_batch_info([], [], chunk=16)
    assert bi["num_segments"] == 0 and bi["seg_indptr"].tolist() == [0]
    bi = oracle.build_batch_info([0, 0], [1, 0], chunk=16)
    assert bi["num_segments"] == 0 and bi["permutation"].size == 0


# --------------------------------------------------------------------------
# shrink / expand / fused
# --------------------------------------------------------------------------

def f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def dense_delta_reference(w: wl.LoraWorkload, base=True):
    """Per token, build the dense weight delta dW_j = sigma * B[off_j:off_j+1, :r] @ A[j*r:(j+1)*r]
    with numpy and apply it to x: (B A) x, the other association order."""
    A, B, x = f64(w.A), f64(w.B), f64(w.x)
    y = f64(w.base).copy() if base else np.zeros((w.s, w.N))
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    for t in range(w.s):
        a = ta[t]
        r = int(w.ranks[a])
        for j in range(w.c):
            o0, o1 = w.offsets[j], w.offsets[j + 1]
            dW = float(w.scalings[a]) * (B[a, o0:o1, :r] @ A[a, j * r:(j + 1) * r, :])
            y[t, o0:o1] += dW @ x[t]
    return y


@pytest.mark.parametrize("seed", range(6))
def test_fused_matches_dense_delta(seed):
    w = wl.random_lora(seed, bs=5, max_len=6, K=40, N_slices=[16, 8, 24][: 1 + seed % 3], R=7, L=4,
                       rank_choices=[1, 3, 5, 7])
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    ref = dense_delta_reference(w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    y0 = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, None)
    np.testing.assert_allclose(y0, dense_delta_reference(w, base=False), rtol=1e-12, atol=1e-12)


def test_single_adapter_is_dense_matmul():
    w = wl.random_lora(7, bs=3, max_len=9, K=64, N_slices=[16, 32], R=8, L=1, rank_choices=[8],
                       zero_rank_prob=0.0, min_len=1)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    X, A, B = f64(w.x), f64(w.A)[0], f64(w.B)[0]
    H = X @ A.T                      # (s, c*R) = (s, 2*8)
    ref = f64(w.base).copy()
    sig = float(w.scalings[0])
    ref[:, 0:16] += sig * H[:, 0:8] @ B[0:16, :].T
    ref[:, 16:48] += sig * H[:, 8:16] @ B[16:48, :].T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_shrink_matches_matmul_and_zero_pads():
    w = wl.random_lora(8, bs=4, max_len=5, K=48, N_slices=[8, 8, 8], R=6, L=3, rank_choices=[2, 5],
                       zero_rank_prob=0.0)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    h = oracle.shrink(w.x, w.A, w.c, ta, w.ranks)
    X, A = f64(w.x), f64(w.A)
    for t in range(w.s):
        a, r = ta[t], int(w.ranks[ta[t]])
        np.testing.assert_allclose(h[t, :3 * r], A[a, :3 * r] @ X[t], rtol=1e-13, atol=1e-14)
        assert np.all(h[t, 3 * r:] == 0.0)


def test_rank_zero_and_no_adapter_leave_base_exact():
    w = wl.random_lora(9, bs=6, max_len=5, K=32, N_slices=[16], R=4, L=3, rank_choices=[4],
                       zero_rank_prob=0.0, min_len=1, pad_value=3.0e4)
    w.ranks[1] = 0
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    rows = ta == 1
    assert rows.any()
    assert np.array_equal(y[rows], f64(w.base)[rows])
    assert not np.array_equal(y[~rows], f64(w.base)[~rows])


def test_columns_outside_slices_untouched():
    w = wl.random_lora(10, bs=3, max_len=4, K=16, N_slices=[8, 16], R=3, L=2, rank_choices=[3],
                       zero_rank_prob=0.0, min_len=1)
    # shift the slices right by 8 inside a 40-column output
    N = 40
    off = np.array([8, 16, 32], np.int32)
    B = np.zeros((w.L, N, w.R), np.uint16)
    B[:, 8:32, :] = w.B
    base = wl.normal_bf16(np.random.default_rng(0), (w.s, N), 1.0)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y = oracle.fused(w.x, w.A, B, off, w.c, ta, w.ranks, w.scalings, base)
    assert np.array_equal(y[:, :8], f64(base)[:, :8]) and np.array_equal(y[:, 32:], f64(base)[:, 32:])


def test_request_order_invariance():
    w = wl.random_lora(11, bs=7, max_len=6, K=24, N_slices=[8, 8], R=5, L=3)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    order = np.random.default_rng(3).permutation(w.bs)
    starts = np.concatenate([[0], np.cumsum(w.req_lens)])
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in order]).astype(int)
    ta2 = oracle.token_adapter(w.req_lens[order], w.req_adapter[order])
    y2 = oracle.fused(w.x[rows], w.A, w.B, w.offsets, w.c, ta2, w.ranks, w.scalings, w.base[rows])
    assert np.array_equal(y2, y[rows])


def test_linear_in_scaling():
    w = wl.random_lora(12, bs=4, max_len=6, K=32, N_slices=[16], R=4, L=2, zero_rank_prob=0.0)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    base = f64(w.base)
    one = np.ones_like(w.scalings)
    d1 = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, one, w.base) - base
    d3 = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, 3 * one, w.base) - base
    np.testing.assert_allclose(d3, 3 * d1, rtol=1e-9, atol=1e-12)


def test_expand_of_shrink_equals_fused():
    w = wl.random_lora(13, bs=5, max_len=7, K=40, N_slices=[8, 16, 8], R=6, L=4)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    h = oracle.shrink(w.x, w.A, w.c, ta, w.ranks)
    y1 = oracle.expand(h, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    y2 = oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base)
    assert np.array_equal(y1, y2)


def test_padding_is_never_read():
    clean = wl.random_lora(14, bs=5, max_len=7, K=40, N_slices=[8, 16], R=6, L=4, rank_choices=[2, 4, 6])
    dirty = wl.random_lora(14, bs=5, max_len=7, K=40, N_slices=[8, 16], R=6, L=4, rank_choices=[2, 4, 6],
                           pad_value=1.0e30)
    ta = oracle.token_adapter(clean.req_lens, clean.req_adapter)
    y1 = oracle.fused(clean.x, clean.A, clean.B, clean.offsets, clean.c, ta, clean.ranks, clean.scalings, clean.base)
    y2 = oracle.fused(dirty.x, dirty.A, dirty.B, dirty.offsets, dirty.c, ta, dirty.ranks, dirty.scalings, dirty.base)
    assert np.array_equal(y1, y2)


# --------------------------------------------------------------------------
# embedding
# --------------------------------------------------------------------------

def test_embedding_is_column_indexing():
    e = wl.embedding_gather(seed=3, n_req=5, req_len=7, V=97, R=6, L=4)
    e.ranks[:] = [6, 3, 0, 1]
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    out, bad = oracle.embedding(e.ids, e.A_emb, ta, e.ranks)
    assert bad == 0
    ref = e.A_emb[ta, :, e.ids]            # (s, R): column ids[t] of A_emb[w_t]
    mask = np.arange(e.R)[None, :] < e.ranks[ta][:, None]
    assert np.array_equal(out, np.where(mask, ref, 0).astype(np.uint16))


def test_embedding_bad_ids_counted():
    e = wl.embedding_gather(seed=4, n_req=2, req_len=3, V=11, R=4, L=2)
    e.ids[1] = 11
    e.ids[4] = -1
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    out, bad = oracle.embedding(e.ids, e.A_emb, ta, e.ranks)
    assert bad == 2 and not out[1].any() and not out[4].any()


# --------------------------------------------------------------------------
# tuple-form B (base_backend.py run_qkv_lora / run_gate_up_lora docstrings)
# --------------------------------------------------------------------------

def qkv_tuple_of(B, offsets):
    """The qkv tuple form of a single (L, N, R) B with slices q, k, v: a q
    buffer (1, L, N_q, R) and one kv buffer (2, L, N_kv, R), as the
    run_qkv_lora docstring lays them out (k and v of equal width)."""
    q = B[None, :, offsets[0]:offsets[1], :].copy()
    kv = np.stack([B[:, offsets[1]:offsets[2], :], B[:, offsets[2]:offsets[3], :]]).copy()
    return q, kv


@pytest.mark.parametrize("seed", range(4))
def test_sliced_b_matches_dense_delta(seed):
    """Per-slice B against the numpy dense per-token weight delta built from
    each slice's own buffer (q / kv tuple for c = 3, two buffers for c = 2)."""
    c = 3 if seed % 2 == 0 else 2
    widths = [16, 8, 8] if c == 3 else [24, 24]
    w = wl.random_lora(40 + seed, bs=5, max_len=6, K=40, N_slices=widths, R=7, L=4, rank_choices=[1, 3, 5, 7])
    off = w.offsets
    if c == 3:
        q, kv = qkv_tuple_of(w.B, off)
        slices = [q[0], kv[0], kv[1]]
    else:
        slices = [w.B[:, off[0]:off[1], :].copy(), w.B[:, off[1]:off[2], :].copy()]
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    A, x = f64(w.A), f64(w.x)
    ref = f64(w.base).copy()
    for t in range(w.s):
        a = ta[t]
        r = int(w.ranks[a])
        for j in range(c):
            Bj = f64(slices[j])
            dW = float(w.scalings[a]) * (Bj[a, :, :r] @ A[a, j * r:(j + 1) * r, :])
            ref[t, off[j]:off[j + 1]] += dW @ x[t]
    y = oracle.fused_sliced(w.x, w.A, slices, off, c, ta, w.ranks, w.scalings, w.base)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_sliced_b_equals_single_tensor():
    """Cutting one (L, N, R) B into its slices gives the single-tensor result
    exactly (same sums in the same order), and so does the expand alone."""
    w = wl.random_lora(9, bs=6, max_len=7, K=48, N_slices=[32, 16, 16], R=8, L=3, rank_choices=[2, 5, 8])
    off = w.offsets
    slices = [w.B[:, off[j]:off[j + 1], :].copy() for j in range(w.c)]
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    y1 = oracle.fused(w.x, w.A, w.B, off, w.c, ta, w.ranks, w.scalings, w.base)
    y2 = oracle.fused_sliced(w.x, w.A, slices, off, w.c, ta, w.ranks, w.scalings, w.base)
    assert np.array_equal(y1, y2)
    h = oracle.shrink(w.x, w.A, w.c, ta, w.ranks)
    e1 = oracle.expand(h, w.B, off, w.c, ta, w.ranks, w.scalings, None)
    e2 = oracle.expand_sliced(h, slices, off, w.c, ta, w.ranks, w.scalings, None)
    assert np.array_equal(e1, e2)


# --------------------------------------------------------------------------
# extra-token embeddings (base_backend.py run_lora_a_embedding,
# run_extra_token_embedding)
# --------------------------------------------------------------------------

def _extra_case(seed, V=37, R=6, L=3, E=5, s=40):
    rng = np.random.default_rng(seed)
    ranks = np.array([6, 3, 0], np.int32)[:L]
    A = wl.normal_bf16(rng, (L, R, V), 1.0)
    extra = wl.normal_bf16(rng, (L, E, R), 1.0)
    ids = rng.integers(0, V + E, size=s).astype(np.int32)
    ta = rng.integers(0, L, size=s).astype(np.int32)
    return ids, A, extra, ta, ranks, V, E


def test_embedding_extra_is_indexing_of_both_tables():
    """ids below V read A_emb's column, ids in [V, V + E) read the extra row,
    both cut at the slot's rank: numpy indexing of the two tables."""
    ids, A, extra, ta, ranks, V, E = _extra_case(3)
    out, bad = oracle.embedding_extra(ids, A, extra, ta, ranks)
    assert bad == 0
    R = A.shape[1]
    for t in range(len(ids)):
        w, r, i = int(ta[t]), int(ranks[ta[t]]), int(ids[t])
        want = np.zeros(R, np.uint16)
        want[:r] = A[w, :r, i] if i < V else extra[w, i - V, :r]
        assert np.array_equal(out[t], want), t
    # without extra ids it is the plain gather
    base_ids = np.where(ids < V, ids, 0).astype(np.int32)
    o1, _ = oracle.embedding_extra(base_ids, A, extra, ta, ranks)
    o2, _ = oracle.embedding(base_ids, A, ta, ranks)
    assert np.array_equal(o1, o2)


def test_embedding_extra_bad_ids_counted():
    ids, A, extra, ta, ranks, V, E = _extra_case(4)
    ids[[2, 5]] = [V + E, -1]
    out, bad = oracle.embedding_extra(ids, A, extra, ta, ranks)
    assert bad == 2 and not out[2].any() and not out[5].any()


def test_extra_token_embedding_replaces_only_extra_rows():
    """Rows of extra tokens become extra[w][id - V] (every column); rows of
    base-vocabulary ids keep their bits."""
    rng = np.random.default_rng(5)
    V, E, D, L, s = 50, 4, 12, 3, 30
    extra = wl.normal_bf16(rng, (L, E, D), 1.0)
    ids = rng.integers(0, V + E, size=s).astype(np.int32)
    ids[:3] = [V, V + E - 1, 7]
    ta = rng.integers(0, L, size=s).astype(np.int32)
    output = wl.normal_bf16(rng, (s, D), 1.0)
    got, bad = oracle.extra_token_embedding(ids, output, extra, V, ta)
    assert bad == 0
    for t in range(s):
        want = extra[ta[t], ids[t] - V] if ids[t] >= V else output[t]
        assert np.array_equal(got[t], want), t
    ids[4] = V + E
    got2, bad2 = oracle.extra_token_embedding(ids, output, extra, V, ta)
    assert bad2 == 1 and np.array_equal(got2[4], output[4])
