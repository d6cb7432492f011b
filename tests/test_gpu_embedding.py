"""Embedding LoRA-A gather against the oracle: bit-exact, rank masking, bad ids."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import build_batch, dev_bf16, dev_f32, dev_i32, host_bits

pytestmark = pytest.mark.gpu


def run(e, ids=None):
    bi = build_batch(e)
    ids = e.ids if ids is None else ids
    out = torch.full((e.s, e.R), 5.0, dtype=torch.bfloat16, device="cuda")
    B.embedding_lora_a(dev_i32(ids), dev_bf16(e.A_emb), e.V, out, bi)
    torch.cuda.synchronize()
    return host_bits(out), bi


@pytest.mark.parametrize("R,ranks", [(8, [8, 3, 0, 5]), (32, [32, 31, 1, 0]), (64, [64, 40, 33, 7]),
                                     (40, [40, 0, 17, 39])])
def test_small_bit_exact(R, ranks):
    e = wl.embedding_gather(seed=R, n_req=7, req_len=45, V=1000, R=R, L=4)
    e.req_lens = np.array([45, 0, 100, 3, 45, 1, 17], np.int32)
    e.ids = np.random.default_rng(R).integers(0, 1000, size=e.s).astype(np.int32)
    e.ranks[:] = ranks
    out, bi = run(e)
    assert bi.device_status() == 0
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding(e.ids, e.A_emb, ta, e.ranks)
    assert bad == 0
    assert np.array_equal(out, ref)


def test_bad_ids_flagged_and_zeroed():
    e = wl.embedding_gather(seed=3, n_req=4, req_len=10, V=500, R=16, L=3)
    ids = e.ids.copy()
    ids[3] = 500
    ids[17] = -2
    out, bi = run(e, ids)
    assert bi.device_status() & 4
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding(ids, e.A_emb, ta, e.ranks)
    assert bad == 2
    assert np.array_equal(out, ref)


def test_embedding_workload_full_size():
    """8192 ids over vocab 128256, rank 32, 32 slots: every output bit-exact."""
    e = wl.embedding_gather()
    out, bi = run(e)
    assert bi.device_status() == 0
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding(e.ids, e.A_emb, ta, e.ranks)
    assert bad == 0 and np.array_equal(out, ref)


def _with_extra(e, E, frac, seed):
    """Replace a fraction of e's ids by extra-token ids in [V, V + E) and draw
    the slots' extra rows (L, E, R)."""
    rng = np.random.default_rng(seed)
    ids = e.ids.copy()
    pick = rng.random(e.s) < frac
    ids[pick] = e.V + rng.integers(0, E, size=int(pick.sum()))
    extra = wl.normal_bf16(rng, (e.L, E, e.R), 0.02)
    return ids, extra


@pytest.mark.parametrize("R,ranks", [(8, [8, 3, 0, 5]), (32, [32, 31, 1, 0]), (40, [40, 0, 17, 39])])
def test_extra_tokens_bit_exact(R, ranks):
    e = wl.embedding_gather(seed=R + 1, n_req=7, req_len=45, V=1000, R=R, L=4)
    e.req_lens = np.array([45, 0, 100, 3, 45, 1, 17], np.int32)
    e.ids = np.random.default_rng(R).integers(0, 1000, size=e.s).astype(np.int32)
    e.ranks[:] = ranks
    ids, extra = _with_extra(e, 9, 0.3, R)
    bi = build_batch(e)
    out = torch.full((e.s, e.R), 5.0, dtype=torch.bfloat16, device="cuda")
    B.embedding_lora_a_extra(dev_i32(ids), dev_bf16(e.A_emb), e.V, dev_bf16(extra), out, bi)
    torch.cuda.synchronize()
    assert bi.device_status() == 0
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding_extra(ids, e.A_emb, extra, ta, e.ranks)
    assert bad == 0 and np.array_equal(host_bits(out), ref)


def test_extra_tokens_full_size_and_bad_ids():
    """The 8192-id workload with 64 extra tokens (10 % of ids) bit-exact; then
    an id past the extra table and a negative id are flagged and zeroed."""
    e = wl.embedding_gather()
    ids, extra = _with_extra(e, 64, 0.1, 7)
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    for bad_ids in (False, True):
        if bad_ids:
            ids[[5, 4000]] = [e.V + 64, -3]
        bi = build_batch(e)
        out = torch.full((e.s, e.R), 5.0, dtype=torch.bfloat16, device="cuda")
        B.embedding_lora_a_extra(dev_i32(ids), dev_bf16(e.A_emb), e.V, dev_bf16(extra), out, bi)
        torch.cuda.synchronize()
        ref, bad = oracle.embedding_extra(ids, e.A_emb, extra, ta, e.ranks)
        assert bad == (2 if bad_ids else 0)
        assert bool(bi.device_status() & 4) == bad_ids
        assert np.array_equal(host_bits(out), ref)


@pytest.mark.parametrize("D", [4096, 100])
def test_extra_token_embedding_rows(D):
    """run_extra_token_embedding: rows of extra tokens of an (s, D) output are
    replaced by their slot's extra rows, every other row keeps its bits."""
    e = wl.embedding_gather(seed=11, n_req=16, req_len=512 if D == 4096 else 40, V=128256, R=8, L=6)
    ids, _ = _with_extra(e, 16, 0.05, 3)
    rng = np.random.default_rng(4)
    extra = wl.normal_bf16(rng, (e.L, 16, D), 0.5)
    output = wl.normal_bf16(rng, (e.s, D), 0.5)
    bi = build_batch(e)
    y = dev_bf16(output)
    B.extra_token_embedding(dev_i32(ids), y, dev_bf16(extra), e.V, bi)
    torch.cuda.synchronize()
    assert bi.device_status() == 0
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.extra_token_embedding(ids, output, extra, e.V, ta)
    assert bad == 0 and np.array_equal(host_bits(y), ref)


def test_token_major_and_segment_kernels_agree():
    """With per-request fields in the batch info the gather is token-major;
    without them it walks the segments.  Both give the oracle's bits, also
    with extra tokens and ragged ranks."""
    e = wl.embedding_gather(seed=21, n_req=9, req_len=70, V=3000, R=40, L=5)
    e.req_lens = np.array([70, 0, 200, 3, 70, 1, 17, 64, 65], np.int32)
    e.ids = np.random.default_rng(4).integers(0, 3000, size=e.s).astype(np.int32)
    e.ranks[:] = [40, 0, 17, 39, 8]
    ids, extra = _with_extra(e, 11, 0.2, 5)
    lens, ad = dev_i32(e.req_lens), dev_i32(e.req_adapter)
    ranks, scal = dev_i32(e.ranks), dev_f32(np.ones(e.L, np.float32))
    outs = []
    for with_req in (True, False):
        bi = B.BatchInfo.for_batch(len(e.req_lens), e.s, e.L, e.R, with_request_fields=with_req)
        B.csgmv_build_batch_info(bi, lens, ad, e.s, ranks, scal)
        out = torch.full((e.s, e.R), 5.0, dtype=torch.bfloat16, device="cuda")
        B.embedding_lora_a_extra(dev_i32(ids), dev_bf16(e.A_emb), e.V, dev_bf16(extra), out, bi)
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        outs.append(host_bits(out))
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding_extra(ids, e.A_emb, extra, ta, e.ranks)
    assert bad == 0
    assert np.array_equal(outs[0], ref) and np.array_equal(outs[1], ref)


def test_transpose_embedding_bit_exact():
    e = wl.embedding_gather(seed=31, n_req=2, req_len=8, V=1000, R=40, L=3)
    At = B.csgmv_transpose_embedding(dev_bf16(e.A_emb))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(At), np.ascontiguousarray(e.A_emb.transpose(0, 2, 1)))


@pytest.mark.parametrize("with_req", [True, False], ids=["token-major", "segments"])
def test_transposed_layout_matches_oracle(with_req):
    """The (L, V, R) table gives the oracle's bits on the (L, R, V) one, with
    extra tokens, ragged and zero ranks and bad ids; and the full-size
    workload bit-exact."""
    e = wl.embedding_gather(seed=32, n_req=7, req_len=45, V=2000, R=24, L=4)
    e.req_lens = np.array([45, 0, 100, 3, 45, 1, 17], np.int32)
    e.ids = np.random.default_rng(6).integers(0, 2000, size=e.s).astype(np.int32)
    e.ranks[:] = [24, 0, 7, 23]
    ids, extra = _with_extra(e, 5, 0.2, 8)
    ids[[3, 50]] = [2005, -1]
    lens, ad = dev_i32(e.req_lens), dev_i32(e.req_adapter)
    bi = B.BatchInfo.for_batch(len(e.req_lens), e.s, e.L, e.R, with_request_fields=with_req)
    B.csgmv_build_batch_info(bi, lens, ad, e.s, dev_i32(e.ranks), dev_f32(np.ones(e.L, np.float32)))
    At = B.csgmv_transpose_embedding(dev_bf16(e.A_emb))
    out = torch.full((e.s, e.R), 5.0, dtype=torch.bfloat16, device="cuda")
    B.embedding_lora_a_transposed(dev_i32(ids), At, e.V, dev_bf16(extra), out, bi)
    torch.cuda.synchronize()
    assert bi.device_status() & 4
    ta = oracle.token_adapter(e.req_lens, e.req_adapter)
    ref, bad = oracle.embedding_extra(ids, e.A_emb, extra, ta, e.ranks)
    assert bad == 2 and np.array_equal(host_bits(out), ref)

    f = wl.embedding_gather()
    bi = build_batch(f)
    At = B.csgmv_transpose_embedding(dev_bf16(f.A_emb))
    out = torch.full((f.s, f.R), 5.0, dtype=torch.bfloat16, device="cuda")
    B.embedding_lora_a_transposed(dev_i32(f.ids), At, f.V, None, out, bi)
    torch.cuda.synchronize()
    ref, bad = oracle.embedding(f.ids, f.A_emb, oracle.token_adapter(f.req_lens, f.req_adapter), f.ranks)
    assert bad == 0 and np.array_equal(host_bits(out), ref)
