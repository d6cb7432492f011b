"""Entry points called first thing in a fresh process: every launcher must
set up what it uses (the tensor-map encoder, kernel attributes) by itself,
not rely on an earlier call of another path."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SNIPPET = r"""
import numpy as np, torch
from segmented_gather_gemm_gb300 import binding as B
from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import build_batch, dev_bf16
w = wl.random_lora(31, bs=3, max_len=500, K=256, N_slices=[128, 128], R=32, L=2, min_len=200)
bi = build_batch(w)
y = dev_bf16(w.base)
{call}
torch.cuda.synchronize()
assert bi.device_status() == 0
print("ok")
"""

CALLS = {
    "qkv_workspace": "ws = torch.empty(B.csgmv_qkv_workspace_bytes(bi, 2) // 4, device='cuda')\n"
                     "B.csgmv_qkv(dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B), w.offsets, 2, 128, y, bi, workspace=ws)",
    "static_scratch": "B.csgmv_qkv_static_scratch(dev_bf16(w.x), dev_bf16(w.A), dev_bf16(w.B), w.offsets, 2, 128, y, bi)",
    "shrink": "h = torch.empty((w.s, 64), dtype=torch.float32, device='cuda')\n"
              "B.csgmv_shrink(dev_bf16(w.x), dev_bf16(w.A), 2, h, bi)",
    "expand": "h = torch.zeros((w.s, 64), dtype=torch.float32, device='cuda')\n"
              "B.csgmv_expand(h, dev_bf16(w.B), w.offsets, 2, 128, y, True, bi)",
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_first_call_in_a_fresh_process(name):
    code = SNIPPET.replace("{call}", CALLS[name])
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.returncode, r.stdout[-2000:], r.stderr[-2000:])
