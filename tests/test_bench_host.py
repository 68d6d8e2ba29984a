"""Host-side bookkeeping of bench.py (no GPU): the algorithmic bytes behind
the roofline figures, the DRAM-traffic file's source check and the
command-line defaults the benchmark contract fixes."""

import os

import bench
from synth import WORKLOADS


def test_algorithmic_bytes_of_the_headline_layer():
    """OPT-13B-shaped layer, batch 1, 8 heads / 1024 neurons, decode
    positions 1024..1151 (mean 1087.5): each entry point's bytes written
    out from the per-unit formulas (selected weights once, the selected
    heads' K/V rows, the inputs, the fp32 output read and written)."""
    w = WORKLOADS["opt13b_stack_fp16"]
    d, dh, r, N, h, s = 5120, 128, 1024, 20480, 40, 2
    assert (w.d, w.d_h, w.r, w.N, w.h) == (d, dh, r, N, h)
    mean_n = w.n_prompt + (w.n_gen - 1) / 2.0
    per = bench._block_bytes(w, 1, mean_n, 8, 1024, 8)
    assert per["mlp"] == 2 * 1024 * d * s + d * s + 8 * d == 21022720
    kv = 8 * 2 * (mean_n + 1) * dh * s
    assert per["attn"] == 8 * 3 * dh * d * s + 8 * dh * d * s + kv + 2 * 8 * dh * s + d * s + 8 * d == 46456832
    assert per["predict"] == (d * r + r * N + d * r + r * h) * s == 62996480
    assert per["ln"] == 4 * d + s * d


def test_batched_bytes_count_the_union_once():
    """At batch B the selected weights of the union are read once; the KV
    rows and the inputs grow with the rows."""
    w = WORKLOADS["opt30b_stack_bf16"]
    one = bench._block_bytes(w, 1, 2047.0, 28, 14336, 28)
    many = bench._block_bytes(w, 32, 2047.0, 28, 14336, 32 * 28)
    weights_mlp = 2 * 14336 * w.d * 2
    assert one["mlp"] - weights_mlp == w.d * 2 + 8 * w.d
    assert many["mlp"] - weights_mlp == 32 * (w.d * 2 + 8 * w.d)
    assert many["predict"] == one["predict"]


def test_traffic_file_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        "# comment = ignored\ncsrc_sha256 = abc123\ndv_sparse_attn = 100\ndv_sparse_mlp = 50\ndv_predict = 7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "_csrc_sha256", lambda: "abc123")
    assert bench._traffic() == {"dv_sparse_attn": 100.0, "dv_sparse_mlp": 50.0, "dv_predict": 7.0}
    monkeypatch.setattr(bench, "_csrc_sha256", lambda: "changed")
    assert bench._traffic() == {}


def test_source_hash_covers_every_kernel_source():
    """Editing any .cu / .cuh / .h under csrc changes the hash (so a stale
    traffic capture is never reported)."""
    csrc = os.path.join(bench.ROOT, "contextual_sparsity_decode_gb300", "csrc")
    names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    assert "k_attn.cu" in names and "tc_common.cuh" in names and "dv_kernels.h" in names
    h = bench._csrc_sha256()
    assert len(h) == 64 and h == bench._csrc_sha256()


def test_contract_defaults():
    a = bench._args([])
    assert (a.gpus, a.impl, a.workload, a.batch) == (1, "ours", "opt13b_stack_fp16", 1)
    assert a.warmup >= 3 and a.steps >= 1
    b = bench._args(["--gpus", "4", "--steps", "7", "--warmup", "3", "--impl", "reference"])
    assert (b.gpus, b.steps, b.warmup, b.impl) == (4, 7, 3, "reference")
