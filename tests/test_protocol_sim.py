"""The runtime protocol on the CPU (mpk_debug_simulate): the real encoded
graphs of the tiny, ~1B, Qwen3-8B-shaped (batch 1: AOT attention; batch 16:
JIT attention) and chained-linear workloads run with one host thread per
worker and per scheduler warp and random task delays, over several steps
(epoch counters are never reset).  Deadlock freedom under hybrid JIT/AOT
and producer-before-consumer order are checked for every task (MPK:
A Compiler and Runtime for Mega-Kernelizing Tensor Programs, §2 Q2 runtime,
Figure 8).  No GPU is used."""
import numpy as np
import pytest

from task_graph_runtime_gb300 import mpk, synth


def _graph(name, workers=148):
    wl = synth.WORKLOADS[name]
    return mpk.Graph(wl.shape, wl.batch, page_size=wl.page_size,
                     max_pages_per_seq=max(1, wl.max_pages_per_seq),
                     num_workers=workers)


def _clean(r, steps):
    assert r["deadlocked"] == 0
    assert r["steps_completed"] == steps
    assert r["order_violations"] == 0
    assert r["duplicate_runs"] == 0
    assert r["missing_runs"] == 0


@pytest.mark.parametrize("name,workers", [
    ("tiny", 3), ("tiny", 17), ("llama1b", 148), ("qwen3_8b", 148),
    ("qwen3_8b_b16", 148), ("chain_b8", 148)])
def test_protocol_completes_in_dependency_order(name, workers):
    g = _graph(name, workers)
    ex = g.export()
    for seed in (1, 2):
        r = g.simulate(steps=3, seed=seed, max_delay_us=8, timeout_ms=60000)
        _clean(r, 3)
        # every task (empty ones included) once per step
        assert r["tasks_run"] == 3 * ex["n_tasks"]
    g.close()


def test_jit_graph_uses_schedulers():
    """Batch 16 puts the attention tasks on the JIT path."""
    g = _graph("qwen3_8b_b16")
    ex = g.export()
    attn = ex["task_kind"] == mpk.TASK_KINDS.index("attn")
    assert (ex["task_launch"][attn] == 1).all()   # MPK_LAUNCH_JIT
    g.close()


def test_unsatisfiable_event_is_reported_as_deadlock():
    g = _graph("tiny", 5)
    ex = g.export()
    first_qkv = int(np.flatnonzero(
        ex["task_kind"] == mpk.TASK_KINDS.index("qkv"))[0])
    g.add_event_count(int(ex["task_dep"][first_qkv]), +1)
    r = g.simulate(steps=1, seed=3, max_delay_us=2, timeout_ms=500)
    assert r["deadlocked"] == 1
    g.close()


def test_undercounted_event_breaks_order():
    """An event that fires one trigger early lets its dependents start
    before a producer has finished; the model must see it."""
    g = _graph("tiny", 5)
    ex = g.export()
    counts = ex["event_count"]
    e = int(np.flatnonzero(counts >= 2)[0])
    g.add_event_count(e, -1)
    r = g.simulate(steps=3, seed=4, max_delay_us=50, timeout_ms=5000)
    assert r["order_violations"] > 0 or r["deadlocked"] == 1
    g.close()
