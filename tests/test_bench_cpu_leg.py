"""The CPU-baseline leg of bench.py on the host (no GPU): the oracle timed on a
bounded sample with the host's BLAS threads, the BLAS library named, and the
one-thread runs in a fresh interpreter."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import bits_plan, get_config, make_expert, make_router, make_shared, make_tokens  # noqa: E402


def test_single_thread_leg_runs_in_a_fresh_interpreter():
    out = bench.cpu_single_thread(names=("tiny",), seconds=0.3, n_tok=2, T=8)
    assert out["threads"] == 1 and out["unit"] == "tokens/s"
    assert isinstance(out["tiny"], float) and out["tiny"] > 0


def test_single_thread_leg_reports_failures():
    out = bench.cpu_single_thread(names=("no-such-layer",), seconds=0.1, n_tok=1, T=2)
    assert out["no-such-layer"].startswith("failed")


def test_cpu_baseline_fields(monkeypatch):
    cfg = get_config("tiny")
    wr, bias = make_router(cfg, 0)
    wl = {"cfg": cfg, "xs": [make_tokens(cfg, 4, 0)], "wr": wr, "bias": bias,
          "experts": [make_expert(cfg, e, 0) for e in range(cfg.E)], "bits": bits_plan(cfg, 0),
          "shared": make_shared(cfg, 0)}
    monkeypatch.setattr(bench, "cpu_single_thread", lambda: {"threads": 1})
    r = bench.cpu_baseline(wl, seconds=0.2)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s" and r["value"] > 0 and r["cores"] >= 1
    assert r["blas"] and r["single_thread"] == {"threads": 1}


def test_algorithmic_bytes_follow_the_byte_model():
    """Bytes a decode step must move: every routed expert's planes at its
    bitwidth (3 d f b / 8) plus its LUT_b rows ((2 f + d) 2^b fp16), or its fp16
    page (3 d f 2); the shared FFN (3 d f_s 2); the step adds the router (d E 2)
    and x in, y out (2 T d 2).  Unrouted experts cost nothing."""
    mix = get_config("mixtral")
    bits = [6, 5, 4, 3, 6, 5, 4, 3]
    off = np.concatenate([[0], np.cumsum([1, 1, 0, 0, 0, 0, 0, 0])])  # one token, experts 0 and 1
    ffn, step = bench.algorithmic_bytes(mix, bits, off, 1)
    d, f = 4096, 14336
    e6 = 3 * d * f * 6 // 8 + (2 * f + d) * 64 * 2
    e5 = 3 * d * f * 5 // 8 + (2 * f + d) * 32 * 2
    assert ffn == e6 + e5 and round(ffn / 1e6, 1) == 248.5
    assert step == ffn + d * 8 * 2 + 2 * 1 * d * 2
    qwen = get_config("qwen")
    bits = [4] + [16] + [3] * 58
    off = np.concatenate([[0], np.cumsum([3, 2] + [0] * 58)])
    ffn, step = bench.algorithmic_bytes(qwen, bits, off, 5)
    b4 = 3 * 2048 * 1408 * 4 // 8 + (2 * 1408 + 2048) * 16 * 2
    assert round(b4 / 1e6, 2) == 4.48
    assert ffn == b4 + 3 * 2048 * 1408 * 2 + 3 * 2048 * 5632 * 2
    assert step == ffn + 2048 * 60 * 2 + 2 * 5 * 2048 * 2


def test_launch_counts_follow_the_library_plan(monkeypatch):
    # the bench's gpu_launches claim: kernels per layer step, from the
    # library's own decode / GEMM split (pw_decode_plan)
    monkeypatch.delenv("PW_DECODE_MAX_TOK", raising=False)
    monkeypatch.delenv("PW_DECODE_MAX_TOK_SHARED", raising=False)
    mix, qwen = get_config("mixtral"), get_config("qwen")
    assert bench._launches_per_step(mix, 8) == 1        # fused step: router to combine in one kernel
    # router, permutation (one kernel up to 1024 slots), row gather, decode kernel, combine
    assert bench._launches_per_step(mix, 64) == 5
    # ... plus the GEMM pair once experts can pass the threshold; two permutation kernels above 1024 slots
    assert bench._launches_per_step(mix, 256) == 7
    assert bench._launches_per_step(mix, 4096) == 8
    # the Qwen-shaped layer's shared FFN leaves the decode kernel above 256 tokens
    assert bench._launches_per_step(qwen, 64) == 5
    assert bench._launches_per_step(qwen, 1024) == 1 + 2 + 1 + 1 + 2 + 2 + 1
