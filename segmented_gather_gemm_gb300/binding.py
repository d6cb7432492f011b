"""ctypes binding of libcsgmv.so (include/csgmv.h), same names as the C ABI.

Argument marshalling only: torch supplies device memory and the current CUDA
stream, every step of the path runs in the library's kernels.  There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsgmv.so")

CSGMV_DTYPE_BF16 = 0
CSGMV_DTYPE_F32 = 1

STATUS_BITS = {
    1: "BAD_ADAPTER", 2: "BAD_RANK", 4: "BAD_TOKEN_ID", 8: "BAD_PERMUTATION", 16: "CAPACITY", 32: "BAD_LENS",
}

EXPORTED = ["csgmv_last_error", "csgmv_version", "csgmv_chunk_size", "csgmv_batch_info_capacity",
            "csgmv_build_batch_info", "csgmv_build_lm_head_batch_info", "csgmv_shrink", "csgmv_expand", "csgmv_qkv", "csgmv_qkv_workspace_bytes",
            "csgmv_qkv_static_scratch", "embedding_lora_a", "embedding_lora_a_extra", "extra_token_embedding",
            "csgmv_expand_sliced", "csgmv_qkv_sliced", "csgmv_qkv_path", "csgmv_tile_table_ints",
            "embedding_lora_a_transposed", "csgmv_transpose_embedding"]

# csgmv_qkv_path results (CSGMV_PATH_*)
PATHS = {0: "fused", 1: "decode", 2: "small_split", 3: "stream"}


class CsgmvError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"csgmv error {code}: {msg}")
        self.code = code


class _BatchInfoC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "seg_indptr", "weight_indices", "permutation", "lora_ranks", "scalings", "num_segments_dev",
        "max_len_dev", "req_seg_indptr", "req_weight_indices", "status")] + [
        (n, ctypes.c_int32) for n in (
            "max_segments", "max_tokens", "max_loras", "max_bs", "max_rank",
            "num_tokens", "chunk_size", "bs", "num_loras", "use_cuda_graph")] + [
        ("tile_table", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded libcsgmv.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with segmented_gather_gemm_gb300.build "
                           "(the csgmv path has no CPU fallback)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    i32p = ctypes.POINTER(ctypes.c_int32)
    bip = ctypes.POINTER(_BatchInfoC)
    sig = {
        "csgmv_last_error": (ctypes.c_char_p, []),
        "csgmv_version": (ctypes.c_char_p, []),
        "csgmv_chunk_size": (i32, [i32, i32]),
        "csgmv_batch_info_capacity": (i32, [i32, i32, i32p, i32p]),
        "csgmv_build_batch_info": (i32, [bip, vp, vp, i32, i32, vp, vp, i32, i32, i32, i32, vp]),
        "csgmv_build_lm_head_batch_info": (i32, [bip, vp, vp, i32, i32, vp, vp, i32, i32, i32, i32, vp]),
        "csgmv_shrink": (i32, [vp, i64, i64, vp, i32, vp, i32, i64, bip, vp]),
        "csgmv_expand": (i32, [vp, i32, i64, vp, i64, i32p, i32, i32, vp, i32, bip, vp]),
        "csgmv_qkv": (i32, [vp, i64, vp, vp, i64, i32p, i32, i32, vp, vp, ctypes.c_size_t, bip, vp]),
        "csgmv_qkv_workspace_bytes": (ctypes.c_size_t, [bip, i32]),
        "csgmv_qkv_static_scratch": (i32, [vp, i64, vp, vp, i64, i32p, i32, i32, vp, bip, vp]),
        "embedding_lora_a": (i32, [vp, vp, i64, i32, vp, bip, vp]),
        "embedding_lora_a_extra": (i32, [vp, vp, i64, i32, vp, i64, vp, bip, vp]),
        "csgmv_expand_sliced": (i32, [vp, i32, i64, ctypes.POINTER(vp), i64, i32p, i32, i32, vp, i32, bip, vp]),
        "csgmv_qkv_sliced": (i32, [vp, i64, vp, ctypes.POINTER(vp), i64, i32p, i32, i32, vp, vp, ctypes.c_size_t,
                                   bip, vp]),
        "extra_token_embedding": (i32, [vp, vp, i64, vp, i64, i64, bip, vp]),
        "csgmv_qkv_path": (i32, [bip, i64, i64, i32p, i32, ctypes.c_size_t]),
        "csgmv_tile_table_ints": (i64, [i32, i32]),
        "embedding_lora_a_transposed": (i32, [vp, vp, i64, i32, vp, i64, vp, bip, vp]),
        "csgmv_transpose_embedding": (i32, [vp, i64, i32, i64, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(rc: int):
    if rc != 0:
        raise CsgmvError(rc, lib().csgmv_last_error().decode())


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _offsets(offsets) -> ctypes.Array:
    vals = [int(v) for v in (offsets.tolist() if hasattr(offsets, "tolist") else offsets)]
    return (ctypes.c_int32 * len(vals))(*vals)


def csgmv_version() -> str:
    return lib().csgmv_version().decode()


def csgmv_chunk_size(num_tokens: int, max_chunk_size: int) -> int:
    return int(lib().csgmv_chunk_size(int(num_tokens), int(max_chunk_size)))


def csgmv_batch_info_capacity(max_bs: int, num_tokens_per_bs: int) -> tuple[int, int]:
    ms, mt = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().csgmv_batch_info_capacity(int(max_bs), int(num_tokens_per_bs), ctypes.byref(ms),
                                           ctypes.byref(mt)))
    return int(ms.value), int(mt.value)


def tile_table_ints(max_loras: int, max_tokens: int) -> int:
    """int32 entries of a batch info's tile table (csgmv_tile_table_ints)."""
    return 4 * (max(max_loras, 0) + max(max_tokens, 0) // 64 + 2)


def csgmv_tile_table_ints(max_loras: int, max_tokens: int) -> int:
    return int(lib().csgmv_tile_table_ints(int(max_loras), int(max_tokens)))


class BatchInfo:
    """Device buffers of one batch info (caller-owned, allocated once by torch)
    plus the C struct that points at them."""

    def __init__(self, max_bs: int, max_tokens: int, max_segments: int, max_loras: int, max_rank: int,
                 device="cuda", with_request_fields: bool = True, with_tile_table: bool = True):
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        self.seg_indptr = torch.zeros(max_segments + 1, **i32)
        self.weight_indices = torch.zeros(max(max_segments, 1), **i32)
        self.permutation = torch.zeros(max(max_tokens, 1), **i32)
        self.lora_ranks = torch.zeros(max_loras, **i32)
        self.scalings = torch.zeros(max_loras, dtype=torch.float32, device=dev)
        self.num_segments = torch.zeros(1, **i32)
        self.max_len = torch.zeros(1, **i32)
        self.status = torch.zeros(1, **i32)
        self.req_seg_indptr = torch.zeros(max_bs + 1, **i32) if with_request_fields else None
        self.req_weight_indices = torch.zeros(max(max_bs, 1), **i32) if with_request_fields else None
        self.tile_table = torch.zeros(tile_table_ints(max_loras, max_tokens), **i32) if with_tile_table else None
        c = _BatchInfoC()
        for n in ("seg_indptr", "weight_indices", "permutation", "lora_ranks", "scalings", "status",
                  "req_seg_indptr", "req_weight_indices", "tile_table"):
            t = getattr(self, n)
            setattr(c, n, t.data_ptr() if t is not None else None)
        c.num_segments_dev = self.num_segments.data_ptr()
        c.max_len_dev = self.max_len.data_ptr()
        c.max_segments, c.max_tokens, c.max_loras = max_segments, max_tokens, max_loras
        c.max_bs, c.max_rank = max_bs, max_rank
        c.num_tokens = -1
        self.c = c

    @classmethod
    def for_cuda_graph(cls, max_bs: int, num_tokens_per_bs: int, max_loras: int, max_rank: int, **kw):
        """Capacities of chunked_backend.py init_cuda_graph_batch_info."""
        ms, mt = csgmv_batch_info_capacity(max_bs, num_tokens_per_bs)
        return cls(max_bs, mt, ms, max_loras, max_rank, **kw)

    @classmethod
    def for_batch(cls, bs: int, num_tokens: int, max_loras: int, max_rank: int, min_chunk: int = 16, **kw):
        """Capacities that fit one eager batch of bs requests and num_tokens
        tokens at any chunk size >= min_chunk: ceil(s / min_chunk) full
        segments plus one partial segment per slot run."""
        ms = (num_tokens + min_chunk - 1) // min_chunk + min(max(bs, 1), max_loras)
        return cls(max(bs, 1), num_tokens, ms, max_loras, max_rank, **kw)

    @property
    def num_tokens(self) -> int:
        return int(self.c.num_tokens)

    @property
    def chunk_size(self) -> int:
        return int(self.c.chunk_size)

    def device_status(self) -> int:
        return int(self.status.item())


def csgmv_build_batch_info(bi: BatchInfo, req_lens: torch.Tensor, req_adapter: torch.Tensor, num_tokens: int,
                           lora_ranks: torch.Tensor, scalings: torch.Tensor, max_chunk_size: int = 128,
                           chunk_size_override: int = 0, use_cuda_graph: bool = False, stream=None) -> None:
    bs = int(req_lens.numel())
    _check(lib().csgmv_build_batch_info(ctypes.byref(bi.c), _ptr(req_lens), _ptr(req_adapter), bs,
                                        int(num_tokens), _ptr(lora_ranks), _ptr(scalings),
                                        int(lora_ranks.numel()), int(max_chunk_size),
                                        int(chunk_size_override), int(bool(use_cuda_graph)), _stream(stream)))


def csgmv_build_lm_head_batch_info(bi: BatchInfo, pruned_lens: torch.Tensor, req_adapter: torch.Tensor,
                                   num_tokens: int, lora_ranks: torch.Tensor, scalings: torch.Tensor,
                                   max_chunk_size: int = 128, chunk_size_override: int = 0,
                                   use_cuda_graph: bool = False, stream=None) -> None:
    bs = int(pruned_lens.numel())
    _check(lib().csgmv_build_lm_head_batch_info(ctypes.byref(bi.c), _ptr(pruned_lens), _ptr(req_adapter), bs,
                                                int(num_tokens), _ptr(lora_ranks), _ptr(scalings),
                                                int(lora_ranks.numel()), int(max_chunk_size),
                                                int(chunk_size_override), int(bool(use_cuda_graph)),
                                                _stream(stream)))


def csgmv_shrink(x: torch.Tensor, A: torch.Tensor, num_slices: int, h: torch.Tensor, bi: BatchInfo,
                 stream=None) -> torch.Tensor:
    s, K = x.shape
    dt = CSGMV_DTYPE_F32 if h.dtype == torch.float32 else CSGMV_DTYPE_BF16
    _check(lib().csgmv_shrink(_ptr(x), int(s), int(K), _ptr(A), int(num_slices), _ptr(h), dt,
                              int(h.stride(0)), ctypes.byref(bi.c), _stream(stream)))
    return h


def csgmv_expand(h: torch.Tensor, B: torch.Tensor, slice_offsets, num_slices: int, max_slice_size: int,
                 out: torch.Tensor, accumulate: bool, bi: BatchInfo, stream=None) -> torch.Tensor:
    dt = CSGMV_DTYPE_F32 if h.dtype == torch.float32 else CSGMV_DTYPE_BF16
    N = int(out.shape[1])
    _check(lib().csgmv_expand(_ptr(h), dt, int(h.stride(0)), _ptr(B), N, _offsets(slice_offsets),
                              int(num_slices), int(max_slice_size), _ptr(out), int(bool(accumulate)),
                              ctypes.byref(bi.c), _stream(stream)))
    return out


def csgmv_qkv(x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, slice_offsets, num_slices: int,
              max_slice_size: int, base_output: torch.Tensor, bi: BatchInfo, stream=None,
              workspace: torch.Tensor | None = None) -> torch.Tensor:
    K = int(x.shape[1])
    N = int(base_output.shape[1])
    ws = _ptr(workspace) if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().csgmv_qkv(_ptr(x), K, _ptr(A), _ptr(B), N, _offsets(slice_offsets), int(num_slices),
                           int(max_slice_size), _ptr(base_output), ws, wsb, ctypes.byref(bi.c), _stream(stream)))
    return base_output


def csgmv_qkv_path(bi: BatchInfo, K: int, N: int, slice_offsets, num_slices: int, workspace_bytes: int) -> str:
    """Which kernels csgmv_qkv runs for the batch last built into bi: "fused"
    (one kernel) or a two-kernel path ("decode", "small_split", "stream").
    Host only."""
    rc = lib().csgmv_qkv_path(ctypes.byref(bi.c), int(K), int(N), _offsets(slice_offsets), int(num_slices),
                              int(workspace_bytes))
    if rc < 0:
        _check(rc)
    return PATHS[rc]


def csgmv_qkv_workspace_bytes(bi: BatchInfo, num_slices: int) -> int:
    return int(lib().csgmv_qkv_workspace_bytes(ctypes.byref(bi.c), int(num_slices)))


def csgmv_qkv_static_scratch(x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, slice_offsets, num_slices: int,
                             max_slice_size: int, base_output: torch.Tensor, bi: BatchInfo,
                             stream=None) -> torch.Tensor:
    """csgmv_qkv with the library's own fixed device scratch for h, for
    callers that cannot allocate a workspace (see csgmv.h)."""
    K = int(x.shape[1])
    N = int(base_output.shape[1])
    _check(lib().csgmv_qkv_static_scratch(_ptr(x), K, _ptr(A), _ptr(B), N, _offsets(slice_offsets),
                                          int(num_slices), int(max_slice_size), _ptr(base_output),
                                          ctypes.byref(bi.c), _stream(stream)))
    return base_output


def embedding_lora_a(input_ids: torch.Tensor, A_emb: torch.Tensor, vocab_size: int, out: torch.Tensor,
                     bi: BatchInfo, stream=None) -> torch.Tensor:
    rank = int(out.shape[1])
    _check(lib().embedding_lora_a(_ptr(input_ids), _ptr(A_emb), int(vocab_size), rank, _ptr(out),
                                  ctypes.byref(bi.c), _stream(stream)))
    return out


def embedding_lora_a_extra(input_ids: torch.Tensor, A_emb: torch.Tensor, vocab_size: int,
                           extra_embeddings: torch.Tensor | None, out: torch.Tensor, bi: BatchInfo,
                           stream=None) -> torch.Tensor:
    """out (s, R) = LoRA-A rows of each token's id, from A_emb (L, R, V) for
    ids below vocab_size and from extra_embeddings (L, E, R) above."""
    E = 0 if extra_embeddings is None else int(extra_embeddings.shape[1])
    _check(lib().embedding_lora_a_extra(_ptr(input_ids), _ptr(A_emb), int(vocab_size), int(out.shape[1]),
                                        _ptr(extra_embeddings), E, _ptr(out), ctypes.byref(bi.c), _stream(stream)))
    return out


def embedding_lora_a_transposed(input_ids: torch.Tensor, A_emb_t: torch.Tensor, vocab_size: int,
                                extra_embeddings: torch.Tensor | None, out: torch.Tensor, bi: BatchInfo,
                                stream=None) -> torch.Tensor:
    """embedding_lora_a_extra with the table stored as A_emb_t (L, V, R)."""
    E = 0 if extra_embeddings is None else int(extra_embeddings.shape[1])
    _check(lib().embedding_lora_a_transposed(_ptr(input_ids), _ptr(A_emb_t), int(vocab_size), int(out.shape[1]),
                                             _ptr(extra_embeddings), E, _ptr(out), ctypes.byref(bi.c),
                                             _stream(stream)))
    return out


def csgmv_transpose_embedding(A_emb: torch.Tensor, A_emb_t: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """A_emb_t (L, V, R) from A_emb (L, R, V), on the device (load time)."""
    L, R, V = (int(v) for v in A_emb.shape)
    if A_emb_t is None:
        A_emb_t = torch.empty((L, V, R), dtype=A_emb.dtype, device=A_emb.device)
    _check(lib().csgmv_transpose_embedding(_ptr(A_emb), L, R, V, _ptr(A_emb_t), _stream(stream)))
    return A_emb_t


def extra_token_embedding(input_ids: torch.Tensor, output: torch.Tensor, extra_embeddings: torch.Tensor,
                          vocab_size: int, bi: BatchInfo, stream=None) -> torch.Tensor:
    """Rows of extra tokens (ids >= vocab_size) of output (s, D) become
    extra_embeddings[slot][id - vocab_size]; other rows are untouched."""
    _check(lib().extra_token_embedding(_ptr(input_ids), _ptr(output), int(output.shape[1]), _ptr(extra_embeddings),
                                       int(extra_embeddings.shape[1]), int(vocab_size), ctypes.byref(bi.c),
                                       _stream(stream)))
    return output


def _slice_ptrs(B_slices) -> ctypes.Array:
    return (ctypes.c_void_p * len(B_slices))(*[t.data_ptr() for t in B_slices])


def csgmv_expand_sliced(h: torch.Tensor, B_slices, slice_offsets, num_slices: int, max_slice_size: int,
                        out: torch.Tensor, accumulate: bool, bi: BatchInfo, stream=None) -> torch.Tensor:
    """csgmv_expand with B given per slice: B_slices[j] is (max_loras, off[j+1]-off[j], R)."""
    dt = CSGMV_DTYPE_F32 if h.dtype == torch.float32 else CSGMV_DTYPE_BF16
    _check(lib().csgmv_expand_sliced(_ptr(h), dt, int(h.stride(0)), _slice_ptrs(B_slices), int(out.shape[1]),
                                     _offsets(slice_offsets), int(num_slices), int(max_slice_size), _ptr(out),
                                     int(bool(accumulate)), ctypes.byref(bi.c), _stream(stream)))
    return out


def csgmv_qkv_sliced(x: torch.Tensor, A: torch.Tensor, B_slices, slice_offsets, num_slices: int,
                     max_slice_size: int, base_output: torch.Tensor, bi: BatchInfo, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """csgmv_qkv with B given per slice (the tuple form of run_qkv_lora /
    run_gate_up_lora): B_slices[j] is (max_loras, off[j+1]-off[j], R)."""
    K = int(x.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().csgmv_qkv_sliced(_ptr(x), K, _ptr(A), _slice_ptrs(B_slices), int(base_output.shape[1]),
                                  _offsets(slice_offsets), int(num_slices), int(max_slice_size), _ptr(base_output),
                                  _ptr(workspace), ws_bytes, ctypes.byref(bi.c), _stream(stream)))
    return base_output
