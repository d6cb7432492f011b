"""The named workloads at their full sizes, in the launch configuration the
benchmark times.  Decode and lm_head are compared element by element; the
prefill workloads on sampled token rows (every column of each sampled row),
which the oracle computes one by one."""
import numpy as np
import pytest

from segmented_gather_gemm_gb300 import workloads as wl
from tests.gpu_helpers import assert_close, f64, oracle_fused, run_fused

pytestmark = pytest.mark.gpu


def sample_rows(w, n=192, seed=0):
    starts = np.concatenate([[0], np.cumsum(w.req_lens)])
    rows = set()
    for i in range(w.bs):  # first and last token of every request
        if w.req_lens[i] > 0:
            rows.add(int(starts[i]))
            rows.add(int(starts[i + 1] - 1))
    rng = np.random.default_rng(seed)
    rows.update(int(t) for t in rng.integers(0, w.s, size=n))
    return np.array(sorted(rows))


def test_decode_qkv_full():
    w = wl.decode_qkv()
    for base in (True, False):
        y, bi = run_fused(w, base=base)
        assert bi.device_status() == 0
        assert_close(f64(y), oracle_fused(w, base=base), f"decode qkv base={base}")


def test_lm_head_decode_full():
    w = wl.lm_head_decode()
    y, bi = run_fused(w)
    assert bi.device_status() == 0
    assert_close(f64(y), oracle_fused(w), "lm_head decode")


@pytest.mark.parametrize("workspace", [False, True], ids=["on-chip", "workspace"])
def test_prefill_gate_up_sampled(workspace):
    """Both csgmv_qkv paths at full size: h on chip, and the two-kernel path
    through a workspace that the bench uses."""
    w = wl.prefill_gate_up()
    rows = sample_rows(w)
    for base in (True, False):
        y, bi = run_fused(w, base=base, workspace=workspace)
        assert bi.device_status() == 0
        assert_close(f64(y[rows]), oracle_fused(w, base=base, rows=rows), f"prefill gate_up base={base}")


def test_skewed_down_proj_chunk_sweep():
    w = wl.skewed_down_proj(chunk=128)
    rows = sample_rows(w)
    ref = oracle_fused(w, rows=rows)
    first = None
    for chunk in (16, 32, 64, 128):
        y, bi = run_fused(w, chunk_override=chunk)
        assert bi.device_status() == 0 and bi.chunk_size == chunk
        assert_close(f64(y[rows]), ref, f"skewed down_proj chunk={chunk}")
        if first is None:
            first = y
        else:
            assert np.array_equal(y, first), "result depends on the chunk size"
