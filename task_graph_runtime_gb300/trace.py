"""Per-task timing of one megakernel step from the device trace
(mpk_debug_set_trace / mpk_debug_read_trace).

  python -m task_graph_runtime_gb300.trace [--workload qwen3_8b] [--steps 3]

Runs `--steps` warm-up steps of the workload (seeded synthetic weights and
KV cache on cuda:0), then one traced step, and prints per task kind the mean
microseconds spent: waiting for its event (``wait``), staging its operands
(``stage``, batch-1 MatMul tiles and attention prologues), on its weight
pages or attention loop (``pages``), in its epilogue, and in its trigger;
then per-worker busy and waiting time.  Tracing adds a global atomic and a
few stores per task, so the step is a little slower than untraced."""
from __future__ import annotations

import argparse
import time

import numpy as np


def summarize(tr: np.ndarray, ex: dict) -> str:
    from . import mpk
    task = (tr[:, 0] & 0xffffffff).astype(np.int64)
    wk = (tr[:, 0] >> 32).astype(np.int64)
    look, ready, staged, pages, body, trig = [tr[:, i].astype(np.int64)
                                              for i in range(1, 7)]
    kinds = ex["task_kind"][task]
    lines = ["%-8s %5s %8s %8s %8s %8s %8s %8s" % (
        "kind", "n", "wait", "stage", "pages", "epilog", "trigger", "exec")]
    for kd in np.unique(kinds):
        m = kinds == kd
        st = np.where(staged[m] > 0, staged[m] - ready[m], 0) / 1e3
        pg = np.where((pages[m] > 0) & (staged[m] > 0),
                      pages[m] - staged[m], 0) / 1e3
        ep = np.where(pages[m] > 0, body[m] - pages[m], 0) / 1e3
        lines.append("%-8s %5d %8.2f %8.2f %8.2f %8.2f %8.2f %8.2f" % (
            mpk.TASK_KINDS[kd], m.sum(), ((ready[m] - look[m]) / 1e3).mean(),
            st.mean(), pg.mean(), ep.mean(),
            ((trig[m] - body[m]) / 1e3).mean(),
            ((trig[m] - ready[m]) / 1e3).mean()))
    busy = np.zeros(wk.max() + 1)
    wait = np.zeros(wk.max() + 1)
    np.add.at(busy, wk, trig - ready)
    np.add.at(wait, wk, ready - look)
    lines.append("per-worker busy ms: mean %.3f min %.3f max %.3f; waiting "
                 "ms: mean %.3f" % (busy.mean() / 1e6, busy.min() / 1e6,
                                    busy.max() / 1e6, wait.mean() / 1e6))
    lines.append("trace span %.3f ms over %d task records" % (
        (trig.max() - look.min()) / 1e6, len(tr)))
    return "\n".join(lines)


def main():
    import torch

    from . import mpk, synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_8b",
                    choices=sorted(synth.WORKLOADS))
    ap.add_argument("--steps", type=int, default=3)
    args = ap.parse_args()
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    W = synth.device_model_weights(s, 0, "cuda")
    g = mpk.Graph(s, wl.batch, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq))
    g.bind(mpk.Weights(W, s))
    kv, seq0 = None, None
    if not s.is_chain:
        k, v, pt, sl = synth.device_kv_inputs(wl, 0, "cuda")
        seq0 = torch.from_numpy(sl).cuda()
        kv = mpk.KVCache(k, v, torch.from_numpy(pt).cuda(), seq0.clone())
    tok = torch.from_numpy(synth.tokens(wl, 0)).cuda()
    lg = torch.empty(wl.batch, s.vocab, device="cuda")
    nt = torch.empty(wl.batch, dtype=torch.int32, device="cuda")

    def step():
        if kv is not None:
            kv.seq_lens.copy_(seq0)
        g.decode_step(tok, kv, lg, nt)

    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    ex = g.export()
    cap = ex["n_tasks"] + 16
    g.set_trace(cap)
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) * 1e3
    tr = g.read_trace(cap)
    if g.status() != mpk.MPK_OK:
        raise RuntimeError(mpk.STATUS_NAMES[g.status()])
    g.close()
    print(f"{args.workload}: traced step wall {wall:.3f} ms")
    print(summarize(tr, ex))


if __name__ == "__main__":
    main()
