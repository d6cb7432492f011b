"""The C-ABI library loads, exports every function include/csgmv.h declares,
and its host-only logic (chunk rule, graph capacities, argument checks that
fail before any CUDA call) behaves as documented.  CPU only: no kernel runs."""
import ctypes
import json
import os
import re

import pytest

from segmented_gather_gemm_gb300 import build as sgb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csgmv.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    try:
        sgb.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    from segmented_gather_gemm_gb300 import binding
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*CSGMV_API\s+(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_][a-z_0-9]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["csgmv_build_batch_info", "csgmv_shrink", "csgmv_expand", "csgmv_qkv", "embedding_lora_a"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from segmented_gather_gemm_gb300 import binding
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in csgmv.h but not exported"
    assert sorted(binding.EXPORTED) == names


def test_chunk_size_matches_rule_table(lib):
    from segmented_gather_gemm_gb300 import binding
    g = json.load(open(os.path.join(GOLDEN, "chunk_size_rule.json")))
    for n, mx, want in g["rows"]:
        assert binding.csgmv_chunk_size(n, mx) == want, (n, mx)


def test_tile_table_size(lib):
    from segmented_gather_gemm_gb300 import binding
    for L, T in ((1, 0), (8, 256), (32, 35509), (256, 2048), (3, 63), (3, 64)):
        assert binding.csgmv_tile_table_ints(L, T) == binding.tile_table_ints(L, T) == 4 * (L + T // 64 + 2)
    assert binding.csgmv_tile_table_ints(-1, 4) == 0


def test_capacity_matches_table(lib):
    from segmented_gather_gemm_gb300 import binding
    g = json.load(open(os.path.join(GOLDEN, "graph_capacity.json")))
    for bs, ntpb, ms, mt in g["rows"]:
        assert binding.csgmv_batch_info_capacity(bs, ntpb) == (ms, mt)
    with pytest.raises(binding.CsgmvError):
        binding.csgmv_batch_info_capacity(-1, 4)
    with pytest.raises(binding.CsgmvError):
        binding.csgmv_batch_info_capacity(1 << 20, 1 << 16)


def _fake_bi(binding, **kw):
    """A batch info whose device pointers are non-NULL placeholders: only
    valid for calls that the host rejects before touching the device."""
    c = binding._BatchInfoC()
    for i, n in enumerate(("seg_indptr", "weight_indices", "permutation", "lora_ranks", "scalings",
                           "num_segments_dev", "max_len_dev", "req_seg_indptr", "req_weight_indices", "status")):
        setattr(c, n, 0x1000 * (i + 1))
    c.max_segments, c.max_tokens, c.max_loras, c.max_bs, c.max_rank = 16, 64, 4, 8, 16
    c.num_tokens, c.chunk_size, c.bs, c.num_loras = 32, 16, 4, 4
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_host_argument_checks(lib):
    from segmented_gather_gemm_gb300 import binding
    INVALID, CAPACITY, UNSUPPORTED = -1, -2, -6
    c = _fake_bi(binding)
    off = (ctypes.c_int32 * 4)(0, 64, 128, 192)
    P = ctypes.c_void_p(0x100000)
    # num_slices outside {1, 2, 3}
    assert lib.csgmv_qkv(P, 64, P, P, 256, off, 4, 64, P, None, 0, ctypes.byref(c), None) == INVALID
    assert b"num_slices" in lib.csgmv_last_error()
    # offsets not multiples of 8
    bad = (ctypes.c_int32 * 2)(0, 60)
    assert lib.csgmv_qkv(P, 64, P, P, 256, bad, 1, 64, P, None, 0, ctypes.byref(c), None) == INVALID
    # max_slice_size below the widest slice
    assert lib.csgmv_qkv(P, 64, P, P, 256, off, 3, 32, P, None, 0, ctypes.byref(c), None) == INVALID
    # offsets beyond N
    assert lib.csgmv_qkv(P, 64, P, P, 128, off, 3, 64, P, None, 0, ctypes.byref(c), None) == INVALID
    # K not a multiple of 8
    assert lib.csgmv_qkv(P, 60, P, P, 256, off, 3, 64, P, None, 0, ctypes.byref(c), None) == INVALID
    # rank above the kernels' limit
    big = _fake_bi(binding, max_rank=128)
    assert lib.csgmv_qkv(P, 64, P, P, 256, off, 3, 64, P, None, 0, ctypes.byref(big), None) == UNSUPPORTED
    # output overlapping the batch info
    ov = ctypes.c_void_p(0x1000)
    assert lib.csgmv_qkv(P, 64, P, P, 256, off, 3, 64, ov, None, 0, ctypes.byref(c), None) == INVALID
    assert b"overlaps" in lib.csgmv_last_error()
    # builder capacities
    assert lib.csgmv_build_batch_info(ctypes.byref(c), P, P, 9, 32, P, P, 4, 128, 0, 0, None) == CAPACITY
    assert lib.csgmv_build_batch_info(ctypes.byref(c), P, P, 4, 65, P, P, 4, 128, 0, 0, None) == CAPACITY
    assert lib.csgmv_build_batch_info(ctypes.byref(c), P, P, 4, 32, P, P, 5, 128, 0, 0, None) == CAPACITY
    # NULL batch info
    assert lib.csgmv_shrink(P, 32, 64, P, 1, P, 0, 16, None, None) == INVALID
    # s disagreeing with the batch
    assert lib.csgmv_shrink(P, 31, 64, P, 1, P, 0, 16, ctypes.byref(c), None) == INVALID
    # embedding rank limits
    assert lib.embedding_lora_a(P, P, 100, 0, P, ctypes.byref(c), None) == UNSUPPORTED
    assert b"rank" in lib.csgmv_last_error()
