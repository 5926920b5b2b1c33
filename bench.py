"""Decode benchmark: ms/token and achieved HBM bandwidth of greedy decode
steps run by the persistent mega-kernel (at batch 1 by default 32 steps a
launch: the decode loop inside one launch; `--steps-per-launch S` to set).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload qwen3_8b] [--mode mega|kpo|kpo_graph]
                  [--steps-per-launch S]

A step is one pass of the whole decode path (every operator of every layer,
lm_head and argmax) for one batch.  Inputs are synthetic and seeded (random
bf16 weights of the workload's shape, a paged KV cache of the configured
context), generated on the device, so the timed region starts with
everything resident in HBM; the weights (15 GB for the Qwen3-8B shape) are
far larger than L2, so no L2 flush is needed between steps.  Every
`workload.steps` steps the sequences rewind to their configured context
(a 4-byte copy per sequence inside the timed region), so every timed step
decodes at the configured context length.

With N > 1 (torchrun), each rank runs an independent replica (the path has
no exchange step); `value` divides the slowest rank's time by all tokens.
`--impl reference` times the CPU oracle (a bounded sample per step) instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from task_graph_runtime_gb300 import synth  # noqa: E402

METRIC = ("decode ms/token at batch 1 and achieved HBM GB/s vs ~8 TB/s "
          "roofline")
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ byte model
def step_bytes(wl: synth.Workload, seq_lens) -> dict:
    """Algorithmic HBM bytes of one decode step at the given cached lengths:
    every weight once, the B embedding rows, the KV cache read over
    positions 0..seq_len (new token included), the new K/V written, the
    logits written.  Activations between operators stay on chip / in L2 and
    are counted too (tiny)."""
    s = wl.shape
    B = wl.batch
    shapes = synth.weight_shapes(s)
    w = 0
    for name, shp in shapes.items():
        if name == "embed":
            continue
        w += int(np.prod(shp)) * 2
    emb = B * s.hidden * 2
    kv_read = kv_write = 0
    if not s.is_chain:
        per_tok = s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2
        kv_read = int(sum((int(n) + 1) * per_tok for n in seq_lens))
        kv_write = B * per_tok
    logits = B * s.vocab * 4
    return {"weights": w, "embed": emb, "kv_read": kv_read,
            "kv_write": kv_write, "logits": logits,
            "total": w + emb + kv_read + kv_write + logits}


def step_flops(wl, seq_lens) -> float:
    s = wl.shape
    params = sum(int(np.prod(shp)) for n, shp in
                 synth.weight_shapes(s).items() if n != "embed")
    f = 2.0 * wl.batch * params
    if not s.is_chain:
        f += 4.0 * sum(int(n) + 1 for n in seq_lens) * s.n_layers * \
            s.n_q_heads * s.head_dim
    return f


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (100 ms)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(1)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        busy = [v for v in sm if mx and v > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- CPU oracle
def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()
             if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


class OracleSample:
    """One layer of the workload's shape plus 1/L of its lm_head on the
    host, run by the oracle; the decode step's time is scaled from it."""

    def __init__(self, wl: synth.Workload, seed: int = 0):
        from oracle import numerics as nx
        self.nx = nx
        self.wl = wl
        s = wl.shape
        self.B = wl.batch
        if s.is_chain:
            self.W = synth.model_weights(s, seed)
            self.scale = 1.0
            self.sample = "the whole chained-linear step"
            return
        one = synth.ModelShape(1, s.hidden, s.n_q_heads, s.n_kv_heads,
                               s.head_dim, s.ffn, s.vocab, s.rms_eps,
                               s.rope_theta, s.qk_norm)
        shapes = synth.weight_shapes(one)
        W = {}
        for name, shp in shapes.items():
            if name in ("embed", "lm_head"):
                continue
            sd = synth.tensor_seed(name, seed)
            if synth._is_norm(name):
                W[name] = synth.normal_bf16(shp, sd, 0.02, 1.0)
            else:
                W[name] = synth.normal_bf16(shp, sd, 0.02)
        rows = max(8, s.vocab // s.n_layers)
        self.lm = synth.normal_bf16((rows, s.hidden),
                                    synth.tensor_seed("lm_head", seed), 0.02)
        self.W = W
        self.one = one
        swl = synth.Workload("sample", one, wl.batch, wl.ctx, wl.page_size, 1)
        self.kv = synth.kv_inputs(swl, seed)
        self.x = synth.normal_bf16((wl.batch, s.hidden),
                                   synth.tensor_seed("x", seed), 1.0)
        self.scale = float(s.n_layers)
        self.sample = (f"1 of {s.n_layers} layers (batch {wl.batch}, "
                       f"context {list(wl.ctx)[:4]}) + {rows} of {s.vocab} "
                       f"lm_head rows, scaled x{s.n_layers}")

    def run_once(self) -> float:
        """Seconds of one sample, scaled to a whole step (the unscaled
        wall time is left in ``self.last_raw``)."""
        nx = self.nx
        t = time.perf_counter()
        if self.wl.shape.is_chain:
            toks = np.zeros(self.B, np.int32)
            nx.decode_step(self.wl.shape, self.W, toks, None, None, None, None)
            self.last_raw = time.perf_counter() - t
            return self.last_raw
        seq = self.kv.seq_lens.copy()
        h = nx.layer_step(self.one, self.W, 0, self.x, self.kv.k_pool,
                          self.kv.v_pool, self.kv.page_table, seq)
        nf = nx.rmsnorm(h, self.W["layer0.ln1"], self.one.rms_eps)
        nx.argmax_lowest(nx.linear(nf, self.lm))
        self.last_raw = time.perf_counter() - t
        return self.last_raw * self.scale


def cpu_baseline(wl, budget_s: float = 12.0) -> dict:
    smp = OracleSample(wl)
    times = []
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or len(times) < 2:
        times.append(smp.run_once())
        if len(times) >= 50:
            break
    v = statistics.median(times) * 1e3 / wl.batch
    return {"value": v, "unit": "ms/token", "cores": _blas_threads(),
            "kind": "oracle", "sample": smp.sample + f"; median of "
            f"{len(times)} samples"}


# --------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    from task_graph_runtime_gb300 import mpk

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    base = synth.WORKLOADS[args.workload]
    s = base.shape
    block = base.steps                       # steps per rewind
    wl = synth.Workload(base.name, s, base.batch, base.ctx, base.page_size,
                        block + 1)
    B = wl.batch
    # inputs resident in HBM
    W = synth.device_model_weights(s, 0, dev)
    g = mpk.Graph(s, B, page_size=wl.page_size,
                  max_pages_per_seq=max(1, wl.max_pages_per_seq))
    g.bind(mpk.Weights(W, s))
    mode = {"mega": mpk.MODE_MEGAKERNEL, "kpo": mpk.MODE_KPO,
            "kpo_graph": mpk.MODE_KPO_GRAPH}[args.mode]
    g.set_mode(mode)
    kv = None
    seq0 = None
    if not s.is_chain:
        k, v, pt, sl = synth.device_kv_inputs(wl, 0, dev)
        seq0 = torch.from_numpy(sl).to(dev)
        kv = mpk.KVCache(k, v, torch.from_numpy(pt).to(dev), seq0.clone())
    toks = [torch.from_numpy(synth.tokens(wl, 0)).to(dev),
            torch.empty(B, dtype=torch.int32, device=dev)]
    logits = torch.empty(B, s.vocab, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ex = g.export()
    # megakernel: several steps a launch (the decode loop inside the kernel);
    # a launch never crosses a rewind of the sequence lengths
    want = args.steps_per_launch or (32 if B == 1 else 1)
    spl = max(1, min(want, block)) if mode == mpk.MODE_MEGAKERNEL else 1
    while block % spl:
        spl -= 1
    nxt_buf = torch.empty(spl, B, dtype=torch.int32, device=dev)

    def rewind(i):
        if kv is not None and i % block == 0:
            kv.seq_lens.copy_(seq0, non_blocking=True)

    def launch(i, m):
        if m == mpk.MODE_KPO_GRAPH:
            # a captured graph replays fixed buffers: feed the next token
            # back with a 4-byte-per-sequence device copy
            g.decode_step(toks[0], kv, logits, toks[1], stream)
            toks[0].copy_(toks[1], non_blocking=True)
        else:
            g.decode_step(toks[i % 2], kv, logits, toks[(i + 1) % 2], stream)

    def launch_block(i):
        """Steps [i, i + spl) in one megakernel launch."""
        g.decode_steps(toks[0], kv, logits, nxt_buf, spl, stream)
        toks[0].copy_(nxt_buf[spl - 1], non_blocking=True)

    def step(i):
        rewind(i)
        launch(i, mode)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        if spl > 1:
            rewind(0)
            launch_block(0)
        torch.cuda.synchronize(dev)
        st = g.status()
        if st != mpk.MPK_OK:
            raise RuntimeError(f"warm-up failed: {mpk.STATUS_NAMES[st]}")
        # per-launch events
        starts = list(range(0, args.steps, spl))
        ev = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in starts]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(local_rank)
        clocks.start()
        time.sleep(0.3)
        start.record(stream)
        for j, i in enumerate(starts):
            rewind(i)
            ev[j][0].record(stream)
            if spl > 1 and i + spl <= args.steps:
                launch_block(i)
            else:
                for k in range(i, min(i + spl, args.steps)):
                    launch(k, mode)
            ev[j][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
    st = g.status()
    if st != mpk.MPK_OK:
        raise RuntimeError(f"timed steps failed: {mpk.STATUS_NAMES[st]}")
    total_ms = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
        torch.distributed.barrier()

    # end to end through the C-ABI with host buffers: tokens h2d from
    # pinned memory, the step, next tokens d2h, every step
    h_tok = torch.from_numpy(synth.tokens(wl, 0)).pin_memory()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    e2e_steps = min(args.steps, 4 * block)
    with torch.cuda.stream(stream):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            if kv is not None and i % block == 0:
                kv.seq_lens.copy_(seq0, non_blocking=True)
            toks[0].copy_(h_tok, non_blocking=True)
            g.decode_step(toks[0], kv, logits, toks[1], stream)
            h_next.copy_(toks[1], non_blocking=True)
            stream.synchronize()
            h_tok.copy_(h_next)
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps

    # the same task bodies launched kernel-per-operator (plain, and replayed
    # from a CUDA Graph), same process and inputs: the comparison point
    compare = {}
    if args.compare and world == 1:
        n_cmp = max(4, min(args.steps, 2 * block))
        for name, m in (("megakernel", mpk.MODE_MEGAKERNEL),
                        ("kpo", mpk.MODE_KPO),
                        ("kpo_graph", mpk.MODE_KPO_GRAPH)):
            if m == mode:
                continue
            g.set_mode(m)
            with torch.cuda.stream(stream):
                for i in range(3):
                    rewind(i)
                    launch(i, m)
                torch.cuda.synchronize(dev)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for i in range(n_cmp):
                    rewind(i)
                    launch(i, m)
                b.record(stream)
                torch.cuda.synchronize(dev)
            if g.status() != mpk.MPK_OK:
                raise RuntimeError(f"{name} steps failed")
            compare[name] = {"ms_per_step": round(a.elapsed_time(b) / n_cmp,
                                                  5),
                             "steps": n_cmp}
        g.set_mode(mode)
    g.close()

    # byte model over one rewind block of steps
    if s.is_chain:
        lens = [[]] * block
    else:
        lens = [[c + j for c in wl.ctx] for j in range(block)]
    by = [step_bytes(wl, L) for L in lens]
    bytes_step = statistics.mean(b["total"] for b in by)
    flops_step = statistics.mean(step_flops(wl, L) for L in lens)
    ms_step = total_ms / args.steps
    launch_avg = statistics.mean(launch_ms)
    peak, peak_kind = measured_peaks()
    # one launch = spl whole steps
    achieved = spl * bytes_step / (launch_avg * 1e-3) / 1e9
    traffic = load_traffic(args.workload, args.mode, spl)
    out = {
        "metric": METRIC,
        "value": round(total_ms / (args.steps * B * world), 5),
        "unit": "ms/token",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random bf16 weights and KV cache, "
                "generated on the device)",
        "config": {"workload": args.workload, "batch": B,
                   "context": list(wl.ctx)[:16], "layers": s.n_layers,
                   "hidden": s.hidden, "vocab": s.vocab,
                   "mode": args.mode, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (weights "
                         f"{by[0]['weights'] / 1e9:.2f} GB)",
                   "rewind_every": block},
        "hbm_gbs": round(bytes_step / (ms_step * 1e-3) / 1e9, 1),
        "frac_of_8tbs": round(bytes_step / (ms_step * 1e-3) / 1e9 /
                              NOMINAL_HBM_GBS, 4),
        "bytes_per_step": int(bytes_step),
        "tflops": round(flops_step / (ms_step * 1e-3) / 1e12, 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind,
                     "kernel": "mpk_megakernel" if args.mode == "mega"
                               else "mpk_kpo_kernel (all launches of a step)",
                     "traffic": traffic},
        "clocks": clk,
        "e2e": {"value": round(e2e_ms / B, 5), "unit": "ms/token",
                "h2d_bytes_per_step": 4 * B, "d2h_bytes_per_step": 4 * B,
                "steps": e2e_steps},
        "gpu_launches": len(starts) if mode == mpk.MODE_MEGAKERNEL
                        else args.steps * ex["n_ops"],
        "steps_per_launch": spl,
        "same_run_modes": compare,
        "graph": {"tasks": ex["n_tasks"], "events": ex["n_events"],
                  "empty_tasks": ex["n_empty"], "workers": ex["n_workers"],
                  "sched_sms": ex["n_sched_sms"],
                  "attn_chunks": ex["attn_chunks"]},
    }
    return out


def load_traffic(workload, mode, steps_per_launch=1):
    """DRAM bytes per launch from the committed ncu summary
    profiles/traffic_<workload>_<mode>.txt ("key: value" lines), if it was
    taken on the current kernel source (else null).  The summary holds the
    bytes of a one-step launch; a launch of S steps moves S times as many
    (every step streams the same weights and cache)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}_{mode}.txt")
    src = os.path.join(ROOT, "task_graph_runtime_gb300", "csrc", "kernels.cu")
    if not os.path.exists(p):
        return None
    d = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith(("#", " ", "|")):
                k, v = line.split(":", 1)
                d[k.strip()] = v.strip()
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if d.get("kernels_sha") != h or "dram_bytes_per_step" not in d:
        return None
    return int(float(d["dram_bytes_per_step"])) * steps_per_launch


def run_reference(args):
    wl = synth.WORKLOADS[args.workload]
    smp = OracleSample(wl)
    for _ in range(args.warmup):
        smp.run_once()
    t, raw = [], []
    for _ in range(args.steps):
        t.append(smp.run_once())
        raw.append(smp.last_raw)
    v = statistics.mean(t) * 1e3 / wl.batch
    cores = _blas_threads()
    # each step runs the bounded sample; ms_per_step is its wall time, and
    # `value` scales it to a whole step of the workload (see `sample`)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3),
            "unit": "ms/token", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(statistics.mean(raw) * 1e3, 3),
            "sample_scale": smp.scale,
            "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded random bf16 weights and KV cache)",
            "config": {"workload": args.workload, "batch": wl.batch,
                       "context": list(wl.ctx)[:16]},
            "cpu_baseline": {"value": round(v, 3), "unit": "ms/token",
                             "cores": cores, "kind": "oracle",
                             "sample": smp.sample},
            "e2e": {"value": round(v, 3), "unit": "ms/token",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=320)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b",
                    choices=sorted(synth.WORKLOADS))
    ap.add_argument("--mode", default="mega",
                    choices=["mega", "kpo", "kpo_graph"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--steps-per-launch", type=int, default=0,
                    help="megakernel: greedy steps per launch (the decode "
                         "loop inside one launch); 1: a launch per step; "
                         "0: 32 at batch 1, 1 above (measured faster)")
    ap.add_argument("--no-compare", dest="compare", action="store_false",
                    help="skip the same-run kernel-per-operator timings")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(synth.WORKLOADS[args.workload])
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
