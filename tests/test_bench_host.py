"""Host-side arithmetic of bench.py (no GPU): the per-block FLOP count behind
the path roofline, the reading of committed ncu summaries, and the summary
of a two-stream timeline."""
import hashlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402
from oracle import dit  # noqa: E402


@pytest.mark.parametrize("name", ["tiny", "t2i", "deep", "video", "large"])
def test_block_flops_counts_every_contraction_of_the_block(name):
    """2 FLOPs per multiply-add of every weight matrix applied to every row
    (from the parameter shapes), plus QK^T and PV per request and head."""
    cfg = synthetic.get_config(name)
    R, T = cfg.requests, cfg.tokens
    M = R * T
    shapes = dict(dit.param_shapes(cfg.hidden, cfg.mlp, cfg.cond_dim))
    gemm = sum(2 * M * shapes[w][0] * shapes[w][1] for w in ("qkv_w", "proj_w", "fc1_w", "fc2_w"))
    d = cfg.hidden // cfg.heads
    attn = R * cfg.heads * (2 * T * T * d) * 2
    ada = 2 * R * shapes["ada_w"][0] * shapes["ada_w"][1]
    assert bench.block_flops(cfg, R, T) == (gemm, attn, ada)
    kf = bench.kernel_flops(cfg, R, T)
    assert sum(kf.values()) == gemm + attn
    assert kf["attention"] == attn


def test_profiled_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "layerwise_weight_offloaded_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k_attention.cu"
    src.write_text("// kernel v1\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "attention_t2i.md").write_text(
        "# summary\n\n| a | b |\n|---|---|\n| x: 1 | y |\n\n"
        f"workload: t2i\nkernel_class: attention\nsource_sha256_16: {digest}\ntraffic_bytes_per_launch: 1234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("attention", "t2i") == (1234, os.path.join("profiles", "attention_t2i.md"))
    assert bench.profiled_traffic("attention", "deep") == (None, None)
    assert bench.profiled_traffic("adaln", "t2i") == (None, None)  # no tracked source
    src.write_text("// kernel v2\n")  # the kernel changed after the capture: no traffic figure
    value, where = bench.profiled_traffic("attention", "t2i")
    assert value is None and where.endswith("(kernel changed since capture)")


def test_timeline_summary_sums_each_stream_and_the_waits():
    ev = [
        {"kernel": "fill", "block": 1, "stream": "copy", "start_ms": 0.0, "end_ms": 0.3},
        {"kernel": "adaln", "block": 1, "stream": "copy", "start_ms": 0.3, "end_ms": 0.35},
        {"kernel": "fill_wait", "block": 0, "stream": "compute", "start_ms": 0.0, "end_ms": 0.01},
        {"kernel": "ln_modulate", "block": 0, "stream": "compute", "start_ms": 0.01, "end_ms": 0.05},
        {"kernel": "attention", "block": 0, "stream": "compute", "start_ms": 0.05, "end_ms": 0.40},
        {"kernel": "fill_wait", "block": 1, "stream": "compute", "start_ms": 0.40, "end_ms": 0.42},
    ]
    got = bench.timeline_summary(ev)
    assert got["span_ms"] == pytest.approx(0.42)
    assert got["copy_busy_ms"] == pytest.approx(0.35)
    assert got["compute_busy_ms"] == pytest.approx(0.39)
    assert got["fill_wait_ms"] == pytest.approx(0.03)
    assert bench.timeline_summary([]) is None
