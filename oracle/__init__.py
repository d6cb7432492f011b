"""CPU oracle for the csgmv multi-adapter LoRA path (TEST INFRASTRUCTURE ONLY).

This package is the slow, plain fp64 reference that the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the product path never does.  It shares no code with
the CUDA library: the arithmetic lives in ``csgmv_oracle.c`` (plain C, OpenMP over
tokens) and this module only marshals numpy arrays into it.

What each function follows (sglang, as printed on the pages):
  chunk_size           chunked_backend.py, _determine_chunk_size_for_tokens
  capacity             chunked_backend.py, init_cuda_graph_batch_info
  token_adapter        chunked_backend.py, _get_permutation (repeat_interleave)
  build_batch_info     chunked_backend.py, prepare_lora_batch / _get_permutation /
                       _get_segments_info / _build_req_seg_indptr
  shrink               base_backend.py, run_lora_a_sgemm; chunked_backend.py,
                       run_lora_a_sgemm (num_slices = c)
  expand               base_backend.py, run_lora_b_sgemm; chunked_backend.py,
                       run_lora_b_sgemm / run_qkv_lora (slice_offsets, base_output)
  fused                chunked_backend.py, run_qkv_lora / run_gate_up_lora
  embedding            base_backend.py, run_lora_a_embedding
  fused_sliced,        base_backend.py, run_qkv_lora / run_gate_up_lora (B as a
  expand_sliced        tuple of per-slice buffers)
  embedding_extra      base_backend.py, run_lora_a_embedding (extra_embeddings)
  extra_token_embedding  base_backend.py, run_extra_token_embedding
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csgmv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile csgmv_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           _SRC, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def use_library(path: str | None):
    """Swap in another build of csgmv_oracle.c (the mutation tests plant
    mistakes in a copy of the source); None restores the normal build."""
    global _lib
    _lib = None if path is None else _bind(ctypes.CDLL(path))


def _bind(lib):
    lib.oracle_chunk_size.restype = ctypes.c_int
    lib.oracle_chunk_size.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.oracle_capacity.restype = None
    lib.oracle_capacity.argtypes = [ctypes.c_int, ctypes.c_int, _i32p, _i32p]
    lib.oracle_token_adapter.restype = ctypes.c_int
    lib.oracle_token_adapter.argtypes = [_i32p, _i32p, ctypes.c_int, _i32p]
    lib.oracle_build_batch_info.restype = ctypes.c_int
    lib.oracle_build_batch_info.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, _i32p, _i32p, _i32p, _i32p, _i32p,
                                            _i32p, _i32p]
    lib.oracle_shrink.restype = ctypes.c_int
    lib.oracle_build_lm_head_batch_info.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, _i32p, _i32p, _i32p, _i32p]
    lib.oracle_build_lm_head_batch_info.restype = ctypes.c_int
    lib.oracle_shrink.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, _u16p, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, _i32p, _i32p, _f64p]
    lib.oracle_expand.restype = ctypes.c_int
    lib.oracle_expand.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _u16p, ctypes.c_int64,
                                  ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _i32p, _i32p,
                                  _f32p, _u16p, _f64p]
    lib.oracle_fused.restype = ctypes.c_int
    lib.oracle_fused.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, _u16p, _u16p,
                                 ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
                                 _i32p, _i32p, _f32p, _u16p, _f64p]
    lib.oracle_embedding.restype = ctypes.c_int
    lib.oracle_embedding.argtypes = [_i32p, ctypes.c_int64, _u16p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int64, _i32p, _i32p, _u16p]
    _u16pp = ctypes.POINTER(_u16p)
    lib.oracle_expand_sliced.restype = ctypes.c_int
    lib.oracle_expand_sliced.argtypes = [_f64p, ctypes.c_int64, ctypes.c_int64, _u16pp, ctypes.c_int64,
                                         ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _i32p, _i32p,
                                         _f32p, _u16p, _f64p]
    lib.oracle_fused_sliced.restype = ctypes.c_int
    lib.oracle_fused_sliced.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, _u16p, _u16pp,
                                        ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
                                        _i32p, _i32p, _f32p, _u16p, _f64p]
    lib.oracle_embedding_extra.restype = ctypes.c_int
    lib.oracle_embedding_extra.argtypes = [_i32p, ctypes.c_int64, _u16p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int64, _u16p, ctypes.c_int64, _i32p, _i32p, _u16p]
    lib.oracle_extra_token_embedding.restype = ctypes.c_int
    lib.oracle_extra_token_embedding.argtypes = [_i32p, ctypes.c_int64, _u16p, ctypes.c_int64, _u16p,
                                                 ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i32p]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray | None, ptype):
    if a is None:
        return ctypes.cast(None, ptype)
    return a.ctypes.data_as(ptype)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def chunk_size(num_tokens: int, max_chunk_size: int) -> int:
    return int(_load().oracle_chunk_size(int(num_tokens), int(max_chunk_size)))


def capacity(max_bs: int, num_tokens_per_bs: int) -> tuple[int, int]:
    ms, mt = ctypes.c_int32(0), ctypes.c_int32(0)
    _load().oracle_capacity(int(max_bs), int(num_tokens_per_bs), ctypes.byref(ms), ctypes.byref(mt))
    return int(ms.value), int(mt.value)


def token_adapter(req_lens, req_adapter) -> np.ndarray:
    lens = _c(req_lens, np.int32)
    ad = _c(req_adapter, np.int32)
    out = np.zeros(max(int(lens.sum()), 1), np.int32)
    n = _load().oracle_token_adapter(_p(lens, _i32p), _p(ad, _i32p), len(lens), _p(out, _i32p))
    return out[:n]


def build_lm_head_batch_info(pruned_lens, req_adapter, chunk: int, use_cuda_graph: bool = False,
                             max_segments: int | None = None) -> dict:
    """Pruned lm_head batch info (identity permutation), as numpy int32 arrays."""
    lens = _c(pruned_lens, np.int32)
    ad = _c(req_adapter, np.int32)
    bs = len(lens)
    s = int(lens.sum())
    if max_segments is None:
        max_segments = max(s, 1)
    perm = np.zeros(max(s, 1), np.int32)
    wi = np.full(max(max_segments, 1), -7, np.int32)
    indptr = np.full(max_segments + 1, -7, np.int32)
    nseg = ctypes.c_int32(0)
    rc = _load().oracle_build_lm_head_batch_info(
        _p(lens, _i32p), _p(ad, _i32p), bs, int(chunk), int(bool(use_cuda_graph)), int(max_segments),
        _p(perm, _i32p), _p(wi, _i32p), _p(indptr, _i32p), ctypes.byref(nseg))
    n = int(nseg.value)
    out = dict(rc=int(rc), num_segments=n, permutation=perm[:s].copy(), chunk=int(chunk), num_tokens=s)
    if use_cuda_graph:
        out["weight_indices"] = wi[:max_segments].copy()
        out["seg_indptr"] = indptr.copy()
    else:
        out["weight_indices"] = wi[:n].copy()
        out["seg_indptr"] = indptr[:n + 1].copy()
    return out


def build_batch_info(req_lens, req_adapter, chunk: int, use_cuda_graph: bool = False,
                     max_segments: int | None = None) -> dict:
    """Batch info of one forward batch, as numpy int32 arrays."""
    lens = _c(req_lens, np.int32)
    ad = _c(req_adapter, np.int32)
    bs = len(lens)
    s = int(lens.sum())
    if max_segments is None:
        max_segments = max(s, 1)
    perm = np.zeros(max(s, 1), np.int32)
    reord = np.zeros(max(s, 1), np.int32)
    wi = np.full(max(max_segments, 1), -7, np.int32)
    indptr = np.full(max_segments + 1, -7, np.int32)
    nseg = ctypes.c_int32(0)
    req_indptr = np.zeros(bs + 1, np.int32)
    req_wi = np.zeros(max(bs, 1), np.int32)
    rc = _load().oracle_build_batch_info(
        _p(lens, _i32p), _p(ad, _i32p), bs, int(chunk), int(bool(use_cuda_graph)),
        int(max_segments), _p(perm, _i32p), _p(reord, _i32p), _p(wi, _i32p), _p(indptr, _i32p),
        ctypes.byref(nseg), _p(req_indptr, _i32p), _p(req_wi, _i32p))
    n = int(nseg.value)
    out = dict(rc=int(rc), num_segments=n, permutation=perm[:s].copy(),
               weights_reordered=reord[:s].copy(), req_seg_indptr=req_indptr,
               req_weight_indices=req_wi[:bs].copy(), chunk=int(chunk), num_tokens=s)
    if use_cuda_graph:
        out["weight_indices"] = wi[:max_segments].copy()
        out["seg_indptr"] = indptr.copy()
    else:
        out["weight_indices"] = wi[:n].copy()
        out["seg_indptr"] = indptr[:n + 1].copy()
    return out


def shrink(x_bits, A_bits, c: int, token_adapter_arr, ranks) -> np.ndarray:
    """h (s, c*R) fp64 from bf16 bit arrays x (s, K) and A (L, c*R, K)."""
    x = _c(x_bits, np.uint16)
    A = _c(A_bits, np.uint16)
    s, K = x.shape
    L, cR, K2 = A.shape
    assert K2 == K and cR % c == 0
    R = cR // c
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    h = np.zeros((s, cR), np.float64)
    _load().oracle_shrink(_p(x, _u16p), s, K, _p(A, _u16p), L, c, R, _p(ta, _i32p),
                          _p(rk, _i32p), _p(h, _f64p))
    return h


def expand(h, B_bits, offsets, c: int, token_adapter_arr, ranks, scalings, base_bits=None) -> np.ndarray:
    """y (s, N) fp64; h is (s, >= c*R) fp64, B (L, N, R) bf16 bits."""
    hh = _c(h, np.float64)
    B = _c(B_bits, np.uint16)
    L, N, R = B.shape
    s = hh.shape[0]
    off = _c(offsets, np.int32)
    assert len(off) == c + 1
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    sc = _c(scalings, np.float32)
    base = None if base_bits is None else _c(base_bits, np.uint16)
    y = np.zeros((s, N), np.float64)
    _load().oracle_expand(_p(hh, _f64p), hh.shape[1], s, _p(B, _u16p), N, L, R, _p(off, _i32p), c,
                          _p(ta, _i32p), _p(rk, _i32p), _p(sc, _f32p), _p(base, _u16p),
                          _p(y, _f64p))
    return y


def fused(x_bits, A_bits, B_bits, offsets, c: int, token_adapter_arr, ranks, scalings,
          base_bits=None) -> np.ndarray:
    """y (s, N) fp64 = base + sigma_w * B_w (A_w x) per slice, h kept in fp64."""
    x = _c(x_bits, np.uint16)
    A = _c(A_bits, np.uint16)
    B = _c(B_bits, np.uint16)
    s, K = x.shape
    L, cR, _ = A.shape
    L2, N, R = B.shape
    assert L2 == L and cR == c * R
    off = _c(offsets, np.int32)
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    sc = _c(scalings, np.float32)
    base = None if base_bits is None else _c(base_bits, np.uint16)
    y = np.zeros((s, N), np.float64)
    _load().oracle_fused(_p(x, _u16p), s, K, _p(A, _u16p), _p(B, _u16p), N, L, R, _p(off, _i32p),
                         c, _p(ta, _i32p), _p(rk, _i32p), _p(sc, _f32p), _p(base, _u16p),
                         _p(y, _f64p))
    return y


def embedding(ids, A_emb_bits, token_adapter_arr, ranks) -> tuple[np.ndarray, int]:
    """(out (s, R) bf16 bits, number of rows with an invalid id or slot)."""
    idv = _c(ids, np.int32)
    A = _c(A_emb_bits, np.uint16)
    L, R, V = A.shape
    s = len(idv)
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    out = np.zeros((s, R), np.uint16)
    bad = _load().oracle_embedding(_p(idv, _i32p), s, _p(A, _u16p), L, R, V, _p(ta, _i32p),
                                   _p(rk, _i32p), _p(out, _u16p))
    return out, int(bad)


def _slice_ptrs(B_slices, c):
    """Per-slice (L, width_j, R) bf16 bit arrays -> (kept arrays, C pointer array, R)."""
    keep = [_c(b, np.uint16) for b in B_slices]
    assert len(keep) == c
    R = keep[0].shape[2]
    arr = (_u16p * c)(*[b.ctypes.data_as(_u16p) for b in keep])
    return keep, arr, R


def expand_sliced(h, B_slices, offsets, c: int, token_adapter_arr, ranks, scalings, base_bits=None) -> np.ndarray:
    """y (s, N) fp64 with B given per slice: B_slices[j] is (L, off[j+1]-off[j], R) bf16 bits."""
    hh = _c(h, np.float64)
    off = _c(offsets, np.int32)
    keep, arr, R = _slice_ptrs(B_slices, c)
    L = keep[0].shape[0]
    N = int(off[-1])
    s = hh.shape[0]
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    sc = _c(scalings, np.float32)
    base = None if base_bits is None else _c(base_bits, np.uint16)
    if base is not None:
        N = base.shape[1]
    y = np.zeros((s, N), np.float64)
    _load().oracle_expand_sliced(_p(hh, _f64p), hh.shape[1], s, arr, N, L, R, _p(off, _i32p), c,
                                 _p(ta, _i32p), _p(rk, _i32p), _p(sc, _f32p), _p(base, _u16p), _p(y, _f64p))
    return y


def fused_sliced(x_bits, A_bits, B_slices, offsets, c: int, token_adapter_arr, ranks, scalings,
                 base_bits=None) -> np.ndarray:
    """y (s, N) fp64 = base + sigma_w * B_j,w (A_w x) per slice j, with B given
    per slice (B_slices[j] of shape (L, off[j+1]-off[j], R)), h kept in fp64."""
    x = _c(x_bits, np.uint16)
    A = _c(A_bits, np.uint16)
    s, K = x.shape
    L, cR, _ = A.shape
    off = _c(offsets, np.int32)
    keep, arr, R = _slice_ptrs(B_slices, c)
    assert cR == c * R
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    sc = _c(scalings, np.float32)
    base = None if base_bits is None else _c(base_bits, np.uint16)
    N = base.shape[1] if base is not None else int(off[-1])
    y = np.zeros((s, N), np.float64)
    _load().oracle_fused_sliced(_p(x, _u16p), s, K, _p(A, _u16p), arr, N, L, R, _p(off, _i32p), c,
                                _p(ta, _i32p), _p(rk, _i32p), _p(sc, _f32p), _p(base, _u16p), _p(y, _f64p))
    return y


def embedding_extra(ids, A_emb_bits, extra_bits, token_adapter_arr, ranks) -> tuple[np.ndarray, int]:
    """(out (s, R) bf16 bits, bad rows) with extra tokens: ids in [V, V + E)
    read extra (L, E, R)."""
    idv = _c(ids, np.int32)
    A = _c(A_emb_bits, np.uint16)
    L, R, V = A.shape
    ex = _c(extra_bits, np.uint16)
    assert ex.shape[0] == L and ex.shape[2] == R
    E = ex.shape[1]
    s = len(idv)
    ta = _c(token_adapter_arr, np.int32)
    rk = _c(ranks, np.int32)
    out = np.zeros((s, R), np.uint16)
    bad = _load().oracle_embedding_extra(_p(idv, _i32p), s, _p(A, _u16p), L, R, V, _p(ex, _u16p), E,
                                         _p(ta, _i32p), _p(rk, _i32p), _p(out, _u16p))
    return out, int(bad)


def extra_token_embedding(ids, output_bits, extra_bits, vocab_size: int, token_adapter_arr) -> tuple[np.ndarray, int]:
    """(output (s, D) bf16 bits with the rows of extra tokens replaced, bad rows)."""
    idv = _c(ids, np.int32)
    out = np.array(output_bits, dtype=np.uint16, copy=True, order="C")
    ex = _c(extra_bits, np.uint16)
    L, E, D = ex.shape
    s = len(idv)
    assert out.shape == (s, D)
    ta = _c(token_adapter_arr, np.int32)
    bad = _load().oracle_extra_token_embedding(_p(idv, _i32p), s, _p(out, _u16p), D, _p(ex, _u16p), L, E,
                                               int(vocab_size), _p(ta, _i32p))
    return out, int(bad)
