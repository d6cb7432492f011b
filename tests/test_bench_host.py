"""Host-side logic of bench.py that the JSON line depends on: the kernel count
per csgmv_qkv call (gpu_launches: the library's own path choice, and the
bench's rule for unbuilt batches checked against it), the algorithmic bytes
of the decode line, and the source hash that keys the recorded DRAM
traffic."""
import os
import shutil

import pytest

import bench
from segmented_gather_gemm_gb300 import workloads as wl


# shapes only (no tensors drawn)
SHAPES = {
    "decode_qkv": lambda: wl.decode_qkv(with_tensors=False),
    "prefill_gate_up": lambda: wl.prefill_gate_up(with_tensors=False),
    "skewed_down_proj": lambda: wl.skewed_down_proj(with_tensors=False),
    "lm_head_decode": lambda: wl.lm_head_decode(with_tensors=False),
    "lm_head_pruned": lambda: wl.lm_head_pruned(with_tensors=False),
    "tiny": wl.tiny_single_slice,
}


@pytest.mark.parametrize("name, kernels", [
    ("decode_qkv", 2),         # 32-token tiles, 6144 columns: the decode shrink and expand
    ("prefill_gate_up", 2),    # 128-token tiles: shrink into the workspace, then expand
    ("skewed_down_proj", 2),   # 128-token tiles, K = 14336: the same two kernels
    ("lm_head_decode", 2),     # 16-token tiles, 128256 columns: the vocabulary-wide split
    ("lm_head_pruned", 2),
    ("tiny", 2),               # 21 tokens per slot: the decode shrink and expand
])
def test_kernels_per_call(name, kernels):
    assert bench.qkv_kernels(SHAPES[name](), None) == kernels


def test_embedding_is_one_kernel():
    assert bench.qkv_kernels(wl.embedding_gather(n_req=2, req_len=4, V=64), None) == 1


@pytest.fixture(scope="module")
def lib():
    from segmented_gather_gemm_gb300 import build as sgb
    try:
        sgb.build()
    except RuntimeError as e:  # no nvcc on this machine
        pytest.skip(str(e))
    from segmented_gather_gemm_gb300 import binding
    return binding


def cpu_batch(B, w, max_segments=None):
    """A batch info with the bench's capacities (max_segments = tokens + 1
    unless given) and the host mirror of workload w, in host memory: enough
    for csgmv_qkv_path, which reads no device buffer."""
    bi = B.BatchInfo(max(w.bs, 1), w.s, w.s + 1 if max_segments is None else max_segments, max_loras=w.L,
                     max_rank=w.R, device="cpu")
    bi.c.num_tokens, bi.c.bs, bi.c.num_loras, bi.c.chunk_size = w.s, w.bs, w.L, 16
    return bi


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_rule_matches_library_path(lib, name):
    w = SHAPES[name]()
    assert bench.qkv_kernels(w, None) == bench.qkv_kernels(w, cpu_batch(lib, w))


def test_library_paths_of_the_workloads(lib):
    want = {"decode_qkv": "decode", "prefill_gate_up": "stream", "skewed_down_proj": "stream",
            "lm_head_decode": "small_split", "lm_head_pruned": "small_split", "tiny": "decode"}
    for name, path in want.items():
        w = SHAPES[name]()
        bi = cpu_batch(lib, w)
        ws = lib.csgmv_qkv_workspace_bytes(bi, w.c)
        assert lib.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, ws) == path, name
        assert lib.csgmv_qkv_path(bi, w.K, w.N, w.offsets, w.c, 0) == "fused", name


def test_small_tile_split_rules(lib):
    """Small tiles take two kernels either way within the decode kernels'
    table capacities; beyond them, only from WIDE_COLS output columns."""
    for cols, kernels, ms in ((bench.WIDE_COLS - 8, 2, None), (bench.WIDE_COLS, 2, None),
                              (bench.WIDE_COLS - 8, 1, 4096), (bench.WIDE_COLS, 2, 4096)):
        w = wl.random_lora(3, bs=40, max_len=1, K=64, N_slices=[cols], R=16, L=6, min_len=1)
        assert bench.qkv_kernels(w, cpu_batch(lib, w, ms)) == kernels
        if ms is None:
            assert bench.qkv_kernels(w, None) == kernels


def test_decode_algorithmic_bytes():
    """x, A and B of the used slots and the base read + write: the decode line's
    13.1 MB (x 2.1 MB, A 3.1 MB, B 1.6 MB, base 2 x 3.1 MB) and its flops."""
    w = wl.decode_qkv(with_tensors=False)
    a = bench.algorithmic(w, 128)
    used = len(set(int(v) for v in w.req_adapter))
    x = w.s * w.K * 2
    A = used * w.c * 16 * w.K * 2
    B = used * w.N * 16 * 2
    base = 2 * w.s * w.N * 2
    assert a["tokens"] == w.s
    assert abs(a["bytes"] - (x + A + B + base)) < 0.01 * (x + A + B + base)
    assert a["flops"] == pytest.approx(w.s * 2 * 16 * (w.c * w.K + w.N), rel=1e-9)


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    """A comment edit keeps the recorded traffic; a code edit drops it."""
    csrc = os.path.join(bench.ROOT, "segmented_gather_gemm_gb300", "csrc")
    root = tmp_path / "repo"
    shutil.copytree(csrc, root / "segmented_gather_gemm_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    f = root / "segmented_gather_gemm_gb300" / "csrc" / "lora_small.cuh"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("#pragma once", "#pragma once  /* note */", 1))
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("#pragma once", "#pragma once\nconstexpr int kUnused = 1;", 1))
    assert bench.kernel_source_hash() != h0


def test_source_hash_is_per_workload(tmp_path, monkeypatch):
    """A change to the small-tile kernel drops the lm_head record but keeps
    the decode and prefill ones, whose kernels do not include it."""
    csrc = os.path.join(bench.ROOT, "segmented_gather_gemm_gb300", "csrc")
    root = tmp_path / "repo"
    shutil.copytree(csrc, root / "segmented_gather_gemm_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    before = {w: bench.kernel_source_hash(w) for w in bench.KERNEL_SOURCES}
    f = root / "segmented_gather_gemm_gb300" / "csrc" / "lora_small.cuh"
    f.write_text(f.read_text().replace("#pragma once", "#pragma once\nconstexpr int kUnused = 1;", 1))
    after = {w: bench.kernel_source_hash(w) for w in bench.KERNEL_SOURCES}
    assert after["prefill_gate_up"] == before["prefill_gate_up"]
    assert after["decode_qkv"] == before["decode_qkv"]
    assert after["lm_head_decode"] != before["lm_head_decode"]
