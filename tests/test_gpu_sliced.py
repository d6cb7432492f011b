"""Tuple-form B (base_backend.py run_qkv_lora: a q buffer (1, L, N_q, R) and a
combined kv buffer (2, L, N_kv, R); run_gate_up_lora: two (L, N, R) buffers),
through csgmv_qkv_sliced and csgmv_expand_sliced.  Each result is compared
with the oracle's per-slice path and must be bit-identical to the
single-tensor call on the same values: decode QKV at full size (16- / 32-token
tiles), prefill-shaped gate_up with and without a workspace (the streaming
shrink + expand, and the fused cluster kernel), and a separate expand."""
import numpy as np
import pytest
import torch

import oracle
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, build_batch, dev_bf16, f64, host_bits

pytestmark = pytest.mark.gpu


def slices_of(w):
    """Per-slice device buffers laid out as the base contract's tuples, and the
    per-slice host arrays for the oracle."""
    off = w.offsets
    host = [np.ascontiguousarray(w.B[:, off[j]:off[j + 1], :]) for j in range(w.c)]
    if w.c == 3:  # q (1, L, N_q, R) and kv (2, L, N_kv, R)
        q = dev_bf16(host[0][None])
        kv = dev_bf16(np.stack([host[1], host[2]]))
        dev = [q[0], kv[0], kv[1]]
        keep = (q, kv)
    else:
        dev = [dev_bf16(h) for h in host]
        keep = tuple(dev)
    return dev, host, keep


def run_both(w, workspace, base=True):
    bi = build_batch(w)
    x, A, Bm = dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B)
    dev, host, keep = slices_of(w)
    widest = int(np.max(np.diff(w.offsets)))
    ws = None
    if workspace:
        ws = torch.full((B.csgmv_qkv_workspace_bytes(bi, w.c) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
    base_bits = w.base if base else np.zeros((w.s, w.N), np.uint16)
    y1, y2 = dev_bf16(base_bits), dev_bf16(base_bits)
    B.csgmv_qkv_sliced(x, A, dev, w.offsets, w.c, widest, y1, bi, workspace=ws)
    B.csgmv_qkv(x, A, Bm, w.offsets, w.c, widest, y2, bi, workspace=ws)
    torch.cuda.synchronize()
    assert bi.device_status() == 0
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    ref = oracle.fused_sliced(w.x, w.A, host, w.offsets, w.c, ta, w.ranks, w.scalings, w.base if base else None)
    return host_bits(y1), host_bits(y2), ref


def test_decode_qkv_tuple_full():
    w = wl.decode_qkv()
    for base in (True, False):
        y1, y2, ref = run_both(w, workspace=True, base=base)
        assert np.array_equal(y1, y2), "tuple-form B differs from the single tensor"
        assert_close(f64(y1), ref, f"decode qkv tuple base={base}")


@pytest.mark.parametrize("workspace", [True, False], ids=["workspace", "on-chip"])
def test_gate_up_tuple_prefill_shape(workspace):
    w = wl.random_lora(21, bs=4, max_len=600, K=320, N_slices=[192, 192], R=32, L=3,
                       rank_choices=list(range(1, 33)), zero_rank_prob=0.2, std=0.5, min_len=150)
    y1, y2, ref = run_both(w, workspace=workspace)
    assert np.array_equal(y1, y2), "tuple-form B differs from the single tensor"
    assert_close(f64(y1), ref, f"gate_up tuple workspace={workspace}")


def test_lm_head_like_tuple_wide():
    """16-token tiles with a vocabulary-wide output split over two slices."""
    w = wl.random_lora(22, bs=40, max_len=1, K=256, N_slices=[16384, 16448], R=16, L=6,
                       rank_choices=[4, 9, 16], zero_rank_prob=0.1, std=0.5, min_len=1)
    y1, y2, ref = run_both(w, workspace=True)
    assert np.array_equal(y1, y2)
    assert_close(f64(y1), ref, "wide tuple")


def test_expand_sliced():
    w = wl.random_lora(23, bs=3, max_len=500, K=128, N_slices=[128, 64, 64], R=64, L=3,
                       rank_choices=[7, 40, 64], zero_rank_prob=0.0, std=0.5, min_len=200)
    bi = build_batch(w)
    ta = oracle.token_adapter(w.req_lens, w.req_adapter)
    href = oracle.shrink(w.x, w.A, w.c, ta, w.ranks)
    h = torch.from_numpy(href.astype(np.float32)).cuda()
    dev, host, keep = slices_of(w)
    for acc in (True, False):
        y = dev_bf16(w.base)
        B.csgmv_expand_sliced(h, dev, w.offsets, w.c, 128, y, acc, bi)
        torch.cuda.synchronize()
        assert bi.device_status() == 0
        ref = oracle.expand_sliced(href, host, w.offsets, w.c, ta, w.ranks, w.scalings, w.base if acc else None)
        assert_close(f64(host_bits(y)), ref, f"expand sliced accumulate={acc}")


def test_sliced_needs_offsets_on_64_columns():
    w = wl.random_lora(24, bs=2, max_len=40, K=64, N_slices=[96, 32], R=16, L=2)
    bi = build_batch(w)
    dev, host, keep = slices_of(w)
    y = dev_bf16(w.base)
    with pytest.raises(B.CsgmvError) as err:
        B.csgmv_qkv_sliced(dev_bf16(w.x), dev_bf16(w.A), dev, w.offsets, w.c, 96, y, bi)
    assert err.value.code == -6
