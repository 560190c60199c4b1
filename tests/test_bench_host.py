"""bench.py's host-side contract, on CPU.

The layer runs on one GPU: it is not sharded and has no collective step, so
a multi-GPU launch (``--gpus N`` with N > 1, or WORLD_SIZE > 1 under
torchrun) must print one "unavailable" line on rank 0, print nothing on the
other ranks, exit 0 and touch no GPU.  The line-building helpers are checked
against hand-computed values.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=env, timeout=300)


@pytest.mark.parametrize("args,env,expect_line", [
    (["--gpus", "2"], {}, True),
    (["--gpus", "8", "--impl", "reference"], {}, True),
    (["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "0"}, True),
    (["--gpus", "2"], {"WORLD_SIZE": "2", "RANK": "1"}, False),
])
def test_multi_gpu_launch_is_refused(args, env, expect_line):
    r = _run(args, env)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if not expect_line:
        assert lines == []
        return
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert "unavailable" in d and "single-GPU" in d["unavailable"]
    assert d["n_gpus"] >= 2


def test_algorithmic_work_of_the_kimi_layer():
    sys.path.insert(0, ROOT)
    import bench
    from mxfp4_weight_moe_gb300 import synthetic as syn

    cfg = syn.CONFIGS["kimi_T8192"]
    w = bench.algorithmic(cfg, 896)
    H, I, T, k = 7168, 3584, 8192, 16
    assert w["layer_flops"] == 6.0 * H * I * T * k
    assert w["w13_bytes_per_expert"] == 2 * I * H // 2 + 2 * I * H // 32
    assert w["w2_bytes_per_expert"] == H * I // 2 + H * I // 32
    assert w["layer_bytes"] == 896 * 1.59375 * H * I + 4 * T * H + 8 * T * k
    c = bench.config_block(cfg, 896, w)
    assert c["workload"].startswith("kimi_T8192") and c["parallelism"] == "single"
    assert set(c) == {"workload", "T", "H", "E", "top_k", "I", "touched_experts", "parallelism", "l2"}


def test_small_layers_are_timed_with_an_l2_flush():
    """Layers whose experts fit in L2 are timed one step at a time with a scrub between steps; the
    gigabyte-scale layers stream their weights from HBM anyway."""
    sys.path.insert(0, ROOT)
    import bench
    from mxfp4_weight_moe_gb300 import synthetic as syn

    for name, flush in (("tiny", True), ("small_T1", True), ("small_T32", True), ("dsv4", False),
                        ("kimi_T16", False), ("kimi_T8192", False)):
        cfg = syn.CONFIGS[name]
        w = bench.algorithmic(cfg, cfg.E)
        assert bench.needs_l2_flush(w) is flush, name
        l2 = bench.config_block(cfg, cfg.E, w)["l2"]
        assert l2.startswith("flushed between steps") is flush, (name, l2)
    assert bench.L2_SCRUB_BYTES > 129e6


def test_timed_ms_scrubs_before_every_call(monkeypatch):
    """With a scrub buffer, the buffer is rewritten before each call and each call has its own event pair."""
    sys.path.insert(0, ROOT)
    import bench

    log = []

    class FakeEvent:
        def __init__(self, enable_timing=False):
            self.t = None

        def record(self, stream=None):
            self.t = len(log)
            log.append("ev")

        def elapsed_time(self, other):
            return float(other.t - self.t)

    class FakeScrub:
        def fill_(self, v):
            log.append("scrub")

    monkeypatch.setattr(bench.torch.cuda, "Event", FakeEvent)
    monkeypatch.setattr(bench.torch.cuda, "synchronize", lambda *a: None)
    ms = bench.timed_ms(lambda i: log.append(f"call{i}"), 3, None, FakeScrub())
    assert log == ["scrub", "ev", "call0", "ev", "scrub", "ev", "call1", "ev", "scrub", "ev", "call2", "ev"]
    assert ms == 3 * 2.0   # each pair brackets exactly its one call
    log.clear()
    ms = bench.timed_ms(lambda i: log.append(f"call{i}"), 2, None, None)
    assert log == ["ev", "call0", "call1", "ev"] and ms == 3.0
