"""Run a few decode steps of a workload, for profiling.

  python -m task_graph_runtime_gb300.run_steps --workload qwen3_8b \
      --mode mega --layers 1 --steps 3 [--coarse]

Seeded synthetic weights and KV cache are generated on cuda:0; `--layers`
keeps only the first N decoder layers (a smaller case of the same kernels,
tiling and launch geometry, for profiler captures that must stay a few GB).
Every step rewinds the sequence lengths, so all steps do the same work.
Prints the device memory in use and the mean step time (CUDA events)."""
from __future__ import annotations

import argparse
import dataclasses


def main():
    import torch

    from . import mpk, synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_8b",
                    choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", default="mega",
                    choices=["mega", "kpo", "kpo_graph"])
    ap.add_argument("--layers", type=int, default=0,
                    help="keep the first N decoder layers (0: all)")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--coarse", action="store_true",
                    help="operator-level events (the coarse-grained graph)")
    args = ap.parse_args()
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    if args.layers > 0 and not s.is_chain:
        s = dataclasses.replace(s, n_layers=min(args.layers, s.n_layers))
        wl = dataclasses.replace(wl, shape=s)
    W = synth.device_model_weights(s, 0, "cuda")
    g = mpk.Graph(s, wl.batch, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq),
                  coarse_events=int(args.coarse))
    g.bind(mpk.Weights(W, s))
    g.set_mode({"mega": mpk.MODE_MEGAKERNEL, "kpo": mpk.MODE_KPO,
                "kpo_graph": mpk.MODE_KPO_GRAPH}[args.mode])
    kv, seq0 = None, None
    if not s.is_chain:
        k, v, pt, sl = synth.device_kv_inputs(wl, 0, "cuda")
        seq0 = torch.from_numpy(sl).cuda()
        kv = mpk.KVCache(k, v, torch.from_numpy(pt).cuda(), seq0.clone())
    tok = torch.from_numpy(synth.tokens(wl, 0)).cuda()
    lg = torch.empty(wl.batch, s.vocab, device="cuda")
    nt = torch.empty(wl.batch, dtype=torch.int32, device="cuda")
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        if kv is not None:
            kv.seq_lens.copy_(seq0)
        g.decode_step(tok, kv, lg, nt)
    e1.record()
    torch.cuda.synchronize()
    if g.status() != mpk.MPK_OK:
        raise RuntimeError(mpk.STATUS_NAMES[g.status()])
    g.close()
    print(f"{args.workload} layers={s.n_layers} mode={args.mode}"
          f"{' coarse' if args.coarse else ''}: "
          f"{e0.elapsed_time(e1) / args.steps:.3f} ms/step, "
          f"{torch.cuda.memory_allocated() / 1e9:.2f} GB on the device")


if __name__ == "__main__":
    main()
