"""Shared helpers of the GPU parity tests: move seeded workloads to the device,
run the library through its C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl

# Tolerance for bf16-in / fp32-accumulate outputs against the fp64 oracle.
RTOL = 1e-2
ATOL = 2e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits_to_f32(host_bits(t)).astype(np.float64)
    return t.detach().cpu().double().numpy()


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "", rtol=RTOL, atol=ATOL):
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside |err| <= {rtol}|ref| + {atol}; "
            f"worst at {worst}: got {got[worst]!r} ref {ref[worst]!r}; first {idx.tolist()}")


def build_batch(w, chunk_override=None, graph=False, capacity=None, stream=None):
    """Batch info on the device for workload w (capacity: (max_bs, ntpb) for graph mode)."""
    s = w.s
    lens = dev_i32(w.req_lens)
    ad = dev_i32(w.req_adapter)
    ranks = dev_i32(w.ranks)
    scal = dev_f32(w.scalings if hasattr(w, "scalings") else np.ones(w.L, np.float32))
    co = w.chunk_override if chunk_override is None else chunk_override
    if capacity is not None:
        bi = B.BatchInfo.for_cuda_graph(capacity[0], capacity[1], max_loras=w.L, max_rank=w.R)
    else:
        bi = B.BatchInfo.for_batch(w.bs if hasattr(w, "bs") else len(w.req_lens), s, w.L, w.R,
                                   min_chunk=min(16, co) if co else 16)
    B.csgmv_build_batch_info(bi, lens, ad, s, ranks, scal, max_chunk_size=w.max_chunk_size,
                             chunk_size_override=co, use_cuda_graph=graph, stream=stream)
    bi._keep = (lens, ad, ranks, scal)
    return bi


def run_fused(w, base=True, chunk_override=None, workspace=False):
    """y = csgmv_qkv on workload w (with a workspace for h if asked);
    returns (y bits, batch info)."""
    bi = build_batch(w, chunk_override)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    y = dev_bf16(w.base) if base else torch.zeros((w.s, w.N), dtype=torch.bfloat16, device="cuda")
    widest = int(np.max(np.diff(w.offsets))) if w.c else 0
    ws = None
    if workspace:
        # filled with NaN: the result must not depend on what it holds
        ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, w.c) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
    B.csgmv_qkv(x, A, Bm, w.offsets, w.c, widest, y, bi, workspace=ws)
    torch.cuda.synchronize()
    return host_bits(y), bi


def oracle_fused(w, base=True, rows=None):
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    if rows is None:
        return oracle.fused(w.x, w.A, w.B, w.offsets, w.c, ta, w.ranks, w.scalings, w.base if base else None)
    return oracle.fused(w.x[rows], w.A, w.B, w.offsets, w.c, ta[rows], w.ranks, w.scalings,
                        w.base[rows] if base else None)


def f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)
