"""Seeded synthetic inputs for the csgmv LoRA path.

This module only draws inputs; it holds none of the method's arithmetic, so the
CUDA library, its tests, the benchmark and the CPU oracle can all take their
inputs from it.  Every tensor is returned as numpy: bf16 tensors as uint16 bit
patterns (fp32 draws rounded to nearest-even), indices as int32.

Draw order inside one generator: request lengths, request adapter slots, slot
ranks, then x, A, B and base (and ids / A_emb for the embedding workload).
Weight rows and columns beyond an adapter's rank (A rows >= c*r_a, B columns
>= r_a) are padding: zero, or ``pad_value`` to check that nothing reads them.

The named workloads follow the shapes of the path's serving scenarios: a tiny
single-slice case, Llama-3-8B-shaped decode QKV, prefill gate_up, skewed
prefill down_proj, and an embedding / lm_head decode case (vocab 128256).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_CHUNK_ELEMS = 1 << 24


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    flat_in = a.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    for lo in range(0, flat_in.size, _CHUNK_ELEMS):
        u = flat_in[lo:lo + _CHUNK_ELEMS].astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        flat_out[lo:lo + _CHUNK_ELEMS] = u.astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std^2) draws in float32, rounded to bf16 bits, drawn in chunks."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, np.uint16)
    for lo in range(0, n, _CHUNK_ELEMS):
        m = min(_CHUNK_ELEMS, n - lo)
        d = rng.standard_normal(m, dtype=np.float32)
        if std != 1.0:
            d *= np.float32(std)
        out[lo:lo + m] = to_bf16_bits(d)
    return out.reshape(shape)


@dataclass
class LoraWorkload:
    """One shrink+expand problem: a batch of requests and the tensors it touches."""
    name: str
    req_lens: np.ndarray          # int32 (bs,)
    req_adapter: np.ndarray       # int32 (bs,)  slot of each request
    ranks: np.ndarray             # int32 (L,)   rank of each slot (0 = no adapter)
    scalings: np.ndarray          # float32 (L,)
    K: int                        # input_dim
    N: int                        # output width (= offsets[-1])
    c: int                        # stacked slices
    R: int                        # max rank (buffer stride)
    offsets: np.ndarray           # int32 (c+1,)
    max_chunk_size: int
    chunk_override: int           # 0 = chunk-size heuristic
    x: np.ndarray | None = None   # bf16 bits (s, K)
    A: np.ndarray | None = None   # bf16 bits (L, c*R, K)
    B: np.ndarray | None = None   # bf16 bits (L, N, R)
    base: np.ndarray | None = None  # bf16 bits (s, N)
    meta: dict = field(default_factory=dict)

    @property
    def bs(self) -> int:
        return int(len(self.req_lens))

    @property
    def s(self) -> int:
        return int(np.sum(self.req_lens))

    @property
    def L(self) -> int:
        return int(len(self.ranks))


@dataclass
class EmbeddingWorkload:
    name: str
    req_lens: np.ndarray
    req_adapter: np.ndarray
    ranks: np.ndarray
    ids: np.ndarray               # int32 (s,)
    A_emb: np.ndarray             # bf16 bits (L, R, V)
    V: int
    R: int
    max_chunk_size: int = 128
    chunk_override: int = 0
    transposed: bool = False      # the table is passed as (L, V, R) (embedding_lora_a_transposed)

    @property
    def s(self) -> int:
        return int(np.sum(self.req_lens))

    @property
    def L(self) -> int:
        return int(len(self.ranks))


def _weights(rng, L, c, R, K, N, ranks, std_a, std_b, pad_value):
    A = normal_bf16(rng, (L, c * R, K), std_a)
    B = normal_bf16(rng, (L, N, R), std_b)
    pad = np.uint16(0) if pad_value is None else to_bf16_bits(np.float32(pad_value)).item()
    for a in range(L):
        r = int(ranks[a])
        A[a, c * r:, :] = pad
        B[a, :, r:] = pad
    return A, B


def _finish(w: LoraWorkload, rng, std_x, std_a, std_b, std_base, pad_value, with_tensors=True):
    if not with_tensors:
        return w
    s = w.s
    w.x = normal_bf16(rng, (s, w.K), std_x)
    w.A, w.B = _weights(rng, w.L, w.c, w.R, w.K, w.N, w.ranks, std_a, std_b, pad_value)
    w.base = normal_bf16(rng, (s, w.N), std_base)
    return w


def tiny_single_slice(seed: int = 0, pad_value=None) -> LoraWorkload:
    """4 requests (7, 16, 25, 16 tokens), K = N = 512, 3 slots of rank 8, 8, 0,
    requests on slots [0, 1, 0, 2], scaling 2.0, N(0, 0.02), chunk 16."""
    rng = np.random.default_rng(seed)
    w = LoraWorkload("tiny_single_slice_s64_k512_n512",
                     req_lens=np.array([7, 16, 25, 16], np.int32),
                     req_adapter=np.array([0, 1, 0, 2], np.int32),
                     ranks=np.array([8, 8, 0], np.int32),
                     scalings=np.full(3, 2.0, np.float32),
                     K=512, N=512, c=1, R=8, offsets=np.array([0, 512], np.int32),
                     max_chunk_size=16, chunk_override=16)
    return _finish(w, rng, 0.02, 0.02, 0.02, 0.02, pad_value)


def decode_qkv(seed: int = 0, bs: int = 256, pad_value=None, with_tensors=True) -> LoraWorkload:
    """Llama-3-8B-shaped decode QKV: bs x 1 token, K = 4096, q 4096 + k 1024 +
    v 1024, c = 3, 8 slots of rank 16 assigned uniformly at random, x ~ N(0, 1),
    A ~ N(0, 1/64^2), B ~ N(0, 1/4^2), base ~ N(0, 1), scaling 2.0."""
    rng = np.random.default_rng(seed)
    L = 8
    lens = np.ones(bs, np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    ranks = np.full(L, 16, np.int32)
    w = LoraWorkload(f"decode_qkv_bs{bs}_k4096_n6144_r16",
                     req_lens=lens, req_adapter=adapter, ranks=ranks,
                     scalings=np.full(L, 2.0, np.float32),
                     K=4096, N=6144, c=3, R=16,
                     offsets=np.array([0, 4096, 5120, 6144], np.int32),
                     max_chunk_size=128, chunk_override=0)
    return _finish(w, rng, 1.0, 1.0 / 64.0, 0.25, 1.0, pad_value, with_tensors)


def prefill_gate_up(seed: int = 0, pad_value=None, with_tensors=True, scale_tokens: float = 1.0) -> LoraWorkload:
    """32 requests of U[64, 2048] tokens, K = 4096, c = 2, 2 x 14336 outputs,
    16 slots with ranks from {8, 16, 32, 64}, Zipf(1.1) slot assignment,
    max_chunk_size 128, N(0, 0.02), scaling 2.0.  ``scale_tokens`` < 1 shrinks
    every request (for small parity cases of the same structure)."""
    rng = np.random.default_rng(seed)
    L = 16
    lens = rng.integers(64, 2049, size=32).astype(np.int32)
    p = (np.arange(L) + 1.0) ** -1.1
    adapter = rng.choice(L, size=32, p=p / p.sum()).astype(np.int32)
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=L).astype(np.int32)
    if scale_tokens != 1.0:
        lens = np.maximum(1, np.round(lens * scale_tokens)).astype(np.int32)
    w = LoraWorkload("prefill_gate_up_k4096_n28672_c2",
                     req_lens=lens, req_adapter=adapter, ranks=ranks,
                     scalings=np.full(L, 2.0, np.float32),
                     K=4096, N=28672, c=2, R=64,
                     offsets=np.array([0, 14336, 28672], np.int32),
                     max_chunk_size=128, chunk_override=0)
    return _finish(w, rng, 0.02, 0.02, 0.02, 0.02, pad_value, with_tensors)


def skewed_down_proj(seed: int = 0, chunk: int = 128, pad_value=None, with_tensors=True,
                     scale_tokens: float = 1.0) -> LoraWorkload:
    """64 requests with Geometric(1/512) lengths, K = 14336, N = 4096, c = 1,
    64 slots of max rank 64 (ranks from {8, 16, ..., 64}), 90 % of requests on
    slot 0 and the rest uniform over slots 1..63, chunk size forced to ``chunk``,
    N(0, 0.02), scaling 2.0."""
    rng = np.random.default_rng(seed)
    L = 64
    lens = rng.geometric(1.0 / 512.0, size=64).astype(np.int32)
    on0 = rng.random(64) < 0.9
    other = rng.integers(1, L, size=64)
    adapter = np.where(on0, 0, other).astype(np.int32)
    ranks = (8 * rng.integers(1, 9, size=L)).astype(np.int32)
    if scale_tokens != 1.0:
        lens = np.maximum(1, np.round(lens * scale_tokens)).astype(np.int32)
    w = LoraWorkload(f"skewed_down_proj_k14336_n4096_chunk{chunk}",
                     req_lens=lens, req_adapter=adapter, ranks=ranks,
                     scalings=np.full(L, 2.0, np.float32),
                     K=14336, N=4096, c=1, R=64,
                     offsets=np.array([0, 4096], np.int32),
                     max_chunk_size=128, chunk_override=int(chunk))
    return _finish(w, rng, 0.02, 0.02, 0.02, 0.02, pad_value, with_tensors)


def lm_head_decode(seed: int = 0, bs: int = 512, pad_value=None, with_tensors=True) -> LoraWorkload:
    """lm_head LoRA decode: bs x 1 token, hidden 4096 -> vocab 128256, c = 1,
    32 slots of rank 32 assigned uniformly, N(0, 0.02), scaling 2.0."""
    rng = np.random.default_rng(seed)
    L = 32
    lens = np.ones(bs, np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    ranks = np.full(L, 32, np.int32)
    w = LoraWorkload(f"lm_head_decode_bs{bs}_k4096_n128256_r32",
                     req_lens=lens, req_adapter=adapter, ranks=ranks,
                     scalings=np.full(L, 2.0, np.float32),
                     K=4096, N=128256, c=1, R=32,
                     offsets=np.array([0, 128256], np.int32),
                     max_chunk_size=128, chunk_override=0)
    return _finish(w, rng, 0.02, 0.02, 0.02, 0.02, pad_value, with_tensors)


def lm_head_pruned(seed: int = 0, bs: int = 64, pad_value=None, with_tensors=True) -> LoraWorkload:
    """Pruned lm_head LoRA after a prefill batch: only the last token of each of
    bs requests reaches lm_head (req_lens holds the pruned token counts, 1 each),
    in request order; hidden 4096 -> vocab 128256, c = 1, 32 slots of rank 32
    assigned uniformly, N(0, 0.02), scaling 2.0.  meta["builder"] = "lm_head":
    the batch info comes from the pruned lm_head builder (identity permutation)."""
    rng = np.random.default_rng(seed)
    L = 32
    lens = np.ones(bs, np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    ranks = np.full(L, 32, np.int32)
    w = LoraWorkload(f"lm_head_pruned_bs{bs}_k4096_n128256_r32",
                     req_lens=lens, req_adapter=adapter, ranks=ranks,
                     scalings=np.full(L, 2.0, np.float32),
                     K=4096, N=128256, c=1, R=32,
                     offsets=np.array([0, 128256], np.int32),
                     max_chunk_size=128, chunk_override=0, meta={"builder": "lm_head"})
    return _finish(w, rng, 0.02, 0.02, 0.02, 0.02, pad_value, with_tensors)


def embedding_gather(seed: int = 0, n_req: int = 16, req_len: int = 512, V: int = 128256,
                     R: int = 32, L: int = 32, pad_value=None) -> EmbeddingWorkload:
    """Embedding LoRA-A: n_req requests of req_len tokens, ids uniform in [0, V),
    L slots of rank R assigned uniformly, A_emb (L, R, V) ~ N(0, 0.02)."""
    rng = np.random.default_rng(seed)
    lens = np.full(n_req, req_len, np.int32)
    adapter = rng.integers(0, L, size=n_req).astype(np.int32)
    ranks = np.full(L, R, np.int32)
    s = int(lens.sum())
    ids = rng.integers(0, V, size=s).astype(np.int32)
    A_emb = normal_bf16(rng, (L, R, V), 0.02)
    if pad_value is not None:
        pad = to_bf16_bits(np.float32(pad_value)).item()
        for a in range(L):
            A_emb[a, int(ranks[a]):, :] = pad
    return EmbeddingWorkload(f"embedding_lora_a_s{s}_v{V}_r{R}", lens, adapter, ranks, ids,
                             A_emb, V, R)


def random_lora(seed: int, bs: int, max_len: int, K: int, N_slices, R: int, L: int,
                rank_choices=None, zero_rank_prob: float = 0.2, std: float = 0.5,
                max_chunk_size: int = 128, chunk_override: int = 0, pad_value=None,
                min_len: int = 0) -> LoraWorkload:
    """Small random case for parity sweeps: ``N_slices`` lists the width of each
    slice (multiples of 8), ranks are drawn from ``rank_choices`` (default
    1..R) with some slots at rank 0, lengths uniform in [min_len, max_len]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len + 1, size=bs).astype(np.int32)
    adapter = rng.integers(0, L, size=bs).astype(np.int32)
    if rank_choices is None:
        rank_choices = np.arange(1, R + 1)
    ranks = rng.choice(np.asarray(rank_choices), size=L).astype(np.int32)
    ranks[rng.random(L) < zero_rank_prob] = 0
    widths = [int(n) for n in N_slices]
    off = np.concatenate([[0], np.cumsum(widths)]).astype(np.int32)
    c = len(widths)
    scal = rng.uniform(0.25, 2.0, size=L).astype(np.float32)
    w = LoraWorkload(f"random_{seed}", lens, adapter, ranks, scal, K=K, N=int(off[-1]), c=c, R=R,
                     offsets=off, max_chunk_size=max_chunk_size, chunk_override=chunk_override)
    return _finish(w, rng, std, std, std, std, pad_value)


WORKLOADS = {
    "tiny": tiny_single_slice,
    "decode_qkv": decode_qkv,
    "prefill_gate_up": prefill_gate_up,
    "skewed_down_proj": skewed_down_proj,
    "lm_head_decode": lm_head_decode,
}
