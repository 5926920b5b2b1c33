"""The C-ABI library on the host (no GPU): it loads, exports every function
include/mpk.h declares, and its C++ tGraph builder reproduces the oracle's
graph bit-exactly (task order, event ids, trigger counts, fan-out ranges,
launch classes, AOT workers)."""
import os
import re

import numpy as np
import pytest

from oracle import tgraph
from task_graph_runtime_gb300 import mpk, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "mpk.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mpk_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mpk_build_tgraph", "mpk_decode_step", "mpk_bind_weights",
              "mpk_export_tgraph", "mpk_get_status", "mpk_reset",
              "mpk_destroy_tgraph", "mpk_set_mode", "mpk_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(mpk_lib):
    missing = [n for n in declared_functions() if not hasattr(mpk_lib, n)]
    assert not missing, missing


def test_status_strings(mpk_lib):
    assert mpk.mpk_status_string(0) == "ok"
    assert "timed out" in mpk.mpk_status_string(6)


def test_invalid_arguments_are_rejected(mpk_lib):
    s = mpk.model_shape(synth.TINY, 16, 9)
    t = mpk.TileSizes(4, 0, 0, 0, 0, 0)
    with pytest.raises(mpk.MpkError) as e:
        mpk.mpk_build_tgraph(s, t, 0)
    assert e.value.status == mpk.MPK_ERR_INVALID_ARG
    bad = mpk.model_shape(synth.ModelShape(2, 256, 4, 3, 64, 688, 1024), 16, 9)
    with pytest.raises(mpk.MpkError):
        mpk.mpk_build_tgraph(bad, t, 1)
    odd = mpk.model_shape(synth.ModelShape(2, 250, 4, 2, 64, 688, 1024), 16, 9)
    with pytest.raises(mpk.MpkError) as e:
        mpk.mpk_build_tgraph(odd, t, 1)
    assert e.value.status == mpk.MPK_ERR_UNSUPPORTED
    with pytest.raises(mpk.MpkError):
        mpk.mpk_build_tgraph(s, mpk.TileSizes(4, 12, 0, 0, 0, 0), 1)
    assert mpk_lib.mpk_decode_step(None, None, None, None, None, None) == \
        mpk.MPK_ERR_INVALID_ARG


CASES = [
    ("tiny_w4", "tiny", 1, dict(num_workers=4)),
    ("tiny_w7", "tiny", 1, dict(num_workers=7)),
    ("tiny_w148", "tiny", 1, dict(num_workers=148)),
    ("tiny_b3_c3", "tiny", 3, dict(num_workers=5, attn_chunks=3)),
    ("tiny_r24", "tiny", 2, dict(num_workers=6, gemv_rows_per_task=24,
                                  attn_chunks=2)),
    ("tiny_c1", "tiny", 1, dict(num_workers=4, attn_chunks=1)),
    ("tiny_coarse", "tiny", 1, dict(num_workers=4, coarse_events=1)),
    ("tiny_b8_mma16", "tiny", 8, dict(num_workers=5, mma_rows_per_task=16)),
    ("llama1b", "llama1b", 1, dict(num_workers=148)),
    ("qwen3_8b", "qwen3_8b", 1, dict(num_workers=148)),
    ("qwen3_8b_b16", "qwen3_8b_b16", 16, dict(num_workers=148)),
    ("chain_b1", "chain_b1", 1, dict(num_workers=148)),
    ("chain_b8", "chain_b8", 8, dict(num_workers=148)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cpp_builder_matches_oracle_builder(mpk_lib, case):
    _, wl_name, B, kw = case
    wl = synth.WORKLOADS[wl_name]
    shape = wl.shape
    page = wl.page_size
    mp = max(1, wl.max_pages_per_seq)
    g = mpk.Graph(shape, B, page_size=page, max_pages_per_seq=mp, **kw)
    ex = g.export()
    g.close()
    ref = tgraph.build(shape, B, mp * page,
                       tgraph.Tiles(kw["num_workers"],
                                    kw.get("gemv_rows_per_task", 0),
                                    kw.get("attn_chunks", 0),
                                    kw.get("mma_rows_per_task", 0),
                                    kw.get("coarse_events", 0)))
    assert ex["n_tasks"] == len(ref.order)
    assert ex["n_events"] == len(ref.ev_count)
    assert ex["n_empty"] == ref.n_empty
    assert ex["n_raw_events"] == len(ref.raw)
    assert ex["n_fused_events"] == len(ref.fused)
    assert ex["attn_chunks"] == ref.n_chunks
    assert np.array_equal(ex["task_pre_id"], ref.order)
    assert np.array_equal(ex["task_dep"], ref.dep)
    assert np.array_equal(ex["task_trig"], ref.trig)
    assert np.array_equal(ex["task_launch"], ref.launch)
    assert np.array_equal(ex["task_worker"], ref.worker)
    assert np.array_equal(ex["event_count"], ref.ev_count)
    assert np.array_equal(ex["event_first"], ref.ev_first)
    assert np.array_equal(ex["event_last"], ref.ev_last)
    kinds = [mpk.TASK_KINDS[k] for k in ex["task_kind"]]
    assert kinds == [ref.tasks[t].kind for t in ref.order]
    for p, t in enumerate(ref.order):
        rt = ref.tasks[t]
        if rt.kind == "empty":
            continue
        assert (ex["task_row0"][p], ex["task_row1"][p]) == (rt.row0, rt.row1)
        assert (ex["task_b"][p], ex["task_g"][p], ex["task_c"][p]) == \
            (rt.b, rt.g, rt.c)
        assert ex["task_tile"][p] == rt.tile
        assert ex["task_layer"][p] == rt.layer
    assert [mpk.TASK_KINDS[k] for k in ex["op_kind"]] == \
        [o.kind for o in ref.ops]
    assert list(ex["op_n_tasks"]) == [o.n_tasks for o in ref.ops]


@pytest.mark.parametrize("name,batch,kw,sched", [
    ("tiny", 1, dict(num_workers=5), 0),              # every task AOT
    ("chain_b8", 8, dict(num_workers=148), 0),        # no attention at all
    ("qwen3_8b_b16", 16, dict(num_workers=148), 4),   # JIT attention
    ("tiny", 1, dict(num_workers=5, num_sched_sms=2, sched_warps_per_sm=3), 2),
])
def test_scheduler_sms_follow_the_jit_tasks(mpk_lib, name, batch, kw, sched):
    """Scheduler SMs default to 4 (Table 1) only when some task is JIT: a
    graph whose tasks are all AOT never dispatches, and a count given
    explicitly is kept."""
    wl = synth.WORKLOADS[name]
    g = mpk.Graph(wl.shape, batch, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq), **kw)
    ex = g.export()
    has_jit = bool((ex["task_launch"] == 1).any())   # MPK_LAUNCH_JIT
    assert ex["n_sched_sms"] == sched
    assert ex["sched_warps_per_sm"] == kw.get("sched_warps_per_sm", 4)
    if "num_sched_sms" not in kw:
        assert (ex["n_sched_sms"] > 0) == has_jit
    assert ex["n_workers"] == kw["num_workers"]
    g.close()
