"""Embedding LoRA-A gather against the oracle: bit-exact, rank masking, bad ids."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import build_batch, dev_bf16, dev_i32, host_bits

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
