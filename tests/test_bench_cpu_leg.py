"""The CPU-baseline leg of bench.py on the host (no GPU): the oracle timed on a
bounded sample with the host's BLAS threads, the BLAS library named, and the
one-thread runs in a fresh interpreter."""
import os
import sys

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
