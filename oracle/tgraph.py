"""Reference tGraph builder.  TEST INFRASTRUCTURE ONLY.

Plain, slow and direct: every set is a Python set and every overlap test a
pairwise comparison of two rectangles.  The steps follow MPK summary, §2 Q2 and §4:

  1. decomposition -- each operator becomes per-output-tile tasks, roughly
     one thread block of work each, about #SMs tasks per operator (MPK
     summary, "Design space & constraint derivation": task granularity;
     MegaKernel HN comments, point 1);
  2. dependencies -- an event for a (producer, consumer) pair iff the
     producer's output region overlaps the consumer's input region (MPK
     summary, §2 Q2 and "6 minimum checks" item 1; MegaKernel HN comments,
     point 2);
  3. event fusion -- successor-set fusion (Def 4.1: equal OutTasks, union
     the InTasks) and predecessor-set fusion (Def 4.2: equal InTasks, union
     the OutTasks), repeated until nothing changes;
  4. normalisation -- every task gets at most one dependent and at most one
     triggering event; each fan-out or fan-in rewrite adds one event and k
     empty tasks (MPK summary, "6 minimum checks" item 3; "关键实现细节" 1);
  5. BFS linearisation -- each event's dependent tasks occupy one contiguous
     index range [first, last] (MPK summary, "6 minimum checks" item 4);
  6. hybrid launch -- attention tasks (data-dependent duration) are JIT,
     the rest AOT (MPK summary, §2 Q2 and "Design space": task launch mode).

Readings taken where the pages are silent:
  * raw events are numbered in (producer id, consumer id) order; a fused
    event keeps the smallest id of its members; S-pass then P-pass, repeated
    to a fixpoint; fusion is not re-applied after normalisation;
  * normalisation rewrites fan-outs first (tasks in ascending id), then
    fan-ins; new tasks and events are numbered after all existing ones in
    creation order;
  * tasks without a dependent event wait on a root event (count 0); tasks
    without a triggering event trigger one end event;
  * linearisation is Kahn-style BFS from the root: a dequeued event's
    OutTasks are appended in ascending pre-linearisation id, and an event is
    enqueued once its last producer has been appended, so the task order is
    also topological;
  * count(e) = |InTasks(e)|;
  * AOT tasks, in linear order, are dealt round-robin to the W workers;
    JIT tasks are placed at run time; empty tasks run inline when their
    event fires;
  * operators of the decode step (a program-level choice the pages leave to
    the compiler): every RMSNorm, with the residual add before it, is the
    prologue of the MatMul that consumes it (each MatMul tile normalises its
    own copy of the input row; tile 0 also stores the residual sum), and the
    query/key RMSNorm, RoPE and KV append are the prologue of the attention
    chunk tasks;
  * split-KV attention: each (sequence, KV head) has C chunk tasks; the
    chunk that finishes last merges the C partials (log-sum-exp), so every
    chunk declares a write of the group's attention output.  Chunks are AOT
    at batch 1 when no chunk can hold more than 128 tokens (equal work,
    known ahead), JIT otherwise (data-dependent lengths).
"""
from __future__ import annotations

import collections
import dataclasses
import math
from typing import Dict, List, Optional, Tuple

# launch classes
AOT, JIT, INLINE = 0, 1, 2

GEMV_KINDS = ("qkv", "o", "gateup", "down", "lm_head", "chain_up",
              "chain_down")
WHOLE = 1 << 30          # a region axis that spans the whole tensor


@dataclasses.dataclass
class Tiles:
    num_workers: int
    gemv_rows_per_task: int = 0     # batch < 8; 0: default split
    attn_chunks: int = 0            # 0: default from the context length
    mma_rows_per_task: int = 0      # batch >= 8; 0: default split
    coarse_events: int = 0          # 1: every read spans its whole tensor


@dataclasses.dataclass
class Task:
    id: int
    op: int                 # index into the op list, -1 for an empty task
    kind: str
    layer: int
    tile: int               # tile index within the op
    row0: int = 0           # GEMV: output rows [row0, row1)
    row1: int = 0
    b: int = 0              # attention family: sequence, KV head, chunk
    g: int = 0
    c: int = 0
    reads: list = dataclasses.field(default_factory=list)
    writes: list = dataclasses.field(default_factory=list)


@dataclasses.dataclass
class Op:
    kind: str
    layer: int
    first_task: int
    n_tasks: int


def tile_row_cap(batch: int, dual: bool, K: int) -> int:
    """Most output rows of one MatMul tile with reduction length K.  Batch 1:
    32 KB pages hold r = max(1, 16384 // K) whole rows; a row's dot product
    is one partial sum when r >= 8, else 8 // r partials, and the tile's
    partials fit 2560 floats.  Batch 2..7: 64 weight rows; batch >= 8: 128.
    A gate/up tile streams two weight rows per output row.  Rounded down to
    a multiple of 8."""
    if batch == 1:
        rpp = max(1, 16384 // K)
        parts = 1 if rpp >= 8 else 8 // rpp
        rows = 2560 // parts
    else:
        rows = 64 if batch < 8 else 128
    if dual:
        rows //= 2
    return max(8, rows // 8 * 8)


def row_tiles(n_rows: int, rows_per_task: int, num_workers: int,
              cap: int, unit: int = 8) -> List[Tuple[int, int]]:
    """Split n_rows output rows into tiles.  Explicit size R: tiles of R
    rows, the last one ragged.  Default: U = ceil(N/unit) units of `unit`
    rows (1 at batch 1, 8 otherwise), T0 = ceil(U / (cap/unit)) tiles at
    least, rounded up to a multiple of the worker count W and clipped to U;
    unit boundaries at floor(i * U / T)."""
    if rows_per_task > 0:
        R = rows_per_task
        return [(s, min(n_rows, s + R)) for s in range(0, n_rows, R)]
    U = -(-n_rows // unit)
    cap_u = max(1, cap // unit)
    T0 = -(-U // cap_u)
    W = max(1, num_workers)
    T = max(1, min(U, W * (-(-T0 // W))))
    out = []
    for i in range(T):
        u0 = (i * U) // T
        u1 = ((i + 1) * U) // T
        out.append((unit * u0, min(n_rows, unit * u1)))
    return out


def default_attn_chunks(batch: int, n_kv_heads: int, max_ctx: int,
                        num_workers: int) -> int:
    by_len = -(-max_ctx // 128)
    by_workers = -(-4 * num_workers // (batch * n_kv_heads))
    return max(1, min(by_len, by_workers))


def attn_is_aot(batch: int, max_ctx: int, chunks: int) -> bool:
    """Chunks of equal, known size (batch 1) that fit 128 tokens."""
    return batch == 1 and chunks > 0 and -(-max_ctx // chunks) <= 128


def decompose(shape, batch: int, max_ctx: int, tiles: Tiles):
    """Operators in program order -> tasks with read/write regions.
    A region is (tensor, r0, r1, c0, c1), a half-open rectangle over a 2-D
    view of the tensor.  With ``tiles.coarse_events`` every read covers its
    whole tensor, so every task of an operator depends on every task of the
    operators it reads (the operator-level graph of Figure 4c)."""
    B = batch
    h, d, F, V = shape.hidden, shape.head_dim, shape.ffn, shape.vocab
    Hq, Hkv = shape.n_q_heads, shape.n_kv_heads
    grp = Hq // Hkv if Hkv else 1
    L = shape.n_layers
    ops: List[Op] = []
    tasks: List[Task] = []

    def rd(tensor, r0, r1, c0, c1):
        if tiles.coarse_events:
            return (tensor, 0, WHOLE, 0, WHOLE)
        return (tensor, r0, r1, c0, c1)

    def add_op(kind, layer, specs):
        op = Op(kind, layer, len(tasks), len(specs))
        for i, sp in enumerate(specs):
            t = Task(id=len(tasks), op=len(ops), kind=kind, layer=layer,
                     tile=i, **sp)
            tasks.append(t)
        ops.append(op)
        return op

    def gemv(kind, layer, n_rows, srcs, dst, k_cols, dual=False, resid=None,
             extra_write=None):
        rpt = tiles.mma_rows_per_task if B >= 8 else tiles.gemv_rows_per_task
        specs = []
        cap = tile_row_cap(B, dual, k_cols)
        if rpt > cap:
            raise ValueError("rows per task above the tile cap")
        tl = row_tiles(n_rows, rpt, tiles.num_workers, cap,
                       1 if B == 1 else 8)
        for i, (r0, r1) in enumerate(tl):
            w = [(dst, 0, B, r0, r1)]
            if i == 0 and resid is not None:
                w.append((resid, 0, B, 0, k_cols))
            if extra_write:
                w.append((extra_write, 0, B, i, i + 1))
            specs.append(dict(row0=r0, row1=r1,
                              reads=[rd(src, 0, B, 0, k_cols) for src in srcs],
                              writes=w))
        return add_op(kind, layer, specs)

    if shape.is_chain:
        # the RMSNorm of the embedding row is W1's prologue
        gemv("chain_up", 0, shape.chain_ffn, [], ("act", 0), h)
        gemv("chain_down", 0, h, [("act", 0)], ("z", 0), shape.chain_ffn)
        lm = gemv("lm_head", 0, V, [("z", 0)], ("logits", 0), h,
                  extra_write=("amax", 0))
        n_chunks = 0
    else:
        C = tiles.attn_chunks or default_attn_chunks(B, Hkv, max_ctx,
                                                     tiles.num_workers)
        n_chunks = C
        for l in range(L):
            srcs = [] if l == 0 else [("hmid", l - 1), ("dout", l - 1)]
            gemv("qkv", l, shape.qkv_rows, srcs, ("qkv", l), h,
                 resid=("h", l))
            specs = []
            for b in range(B):
                for g in range(Hkv):
                    qc = (g * grp * d, (g + 1) * grp * d)
                    kc = (Hq * d + g * d, Hq * d + (g + 1) * d)
                    vc = ((Hq + Hkv) * d + g * d, (Hq + Hkv) * d + (g + 1) * d)
                    for c in range(C):
                        specs.append(dict(
                            b=b, g=g, c=c,
                            reads=[rd(("qkv", l), b, b + 1, *qc),
                                   rd(("qkv", l), b, b + 1, *kc),
                                   rd(("qkv", l), b, b + 1, *vc)],
                            writes=[(("opart", l), b * Hkv + g,
                                     b * Hkv + g + 1, c, c + 1),
                                    (("attn", l), b, b + 1) + qc]))
            add_op("attn", l, specs)
            gemv("o", l, h, [("attn", l)], ("o", l), Hq * d)
            gemv("gateup", l, F, [("h", l), ("o", l)], ("act", l), h,
                 dual=True, resid=("hmid", l))
            gemv("down", l, h, [("act", l)], ("dout", l), F)
        lm = gemv("lm_head", L, V, [("hmid", L - 1), ("dout", L - 1)],
                  ("logits", 0), h, resid=("h", L), extra_write=("amax", 0))
    add_op("argmax", L, [dict(
        reads=[rd(("amax", 0), 0, B, 0, lm.n_tasks)],
        writes=[(("next", 0), 0, B, 0, 1)])])
    return ops, tasks, n_chunks


def _overlap(a, b) -> bool:
    return (a[0] == b[0] and a[1] < b[2] and b[1] < a[2]
            and a[3] < b[4] and b[3] < a[4])


def raw_events(tasks: List[Task]) -> List[Tuple[int, int]]:
    """Every (producer, consumer) pair whose write and read regions overlap;
    sorted by (producer, consumer).  Brute force over every writer/reader
    pair of each tensor (regions of different tensors never overlap)."""
    writers = collections.defaultdict(list)
    readers = collections.defaultdict(list)
    for t in tasks:
        for w in t.writes:
            writers[w[0]].append((t.id, w))
        for r in t.reads:
            readers[r[0]].append((t.id, r))
    pairs = set()
    for key, ws in writers.items():
        for p, w in ws:
            for c, r in readers.get(key, ()):
                if p != c and _overlap(w, r):
                    pairs.add((p, c))
    return sorted(pairs)


def raw_events_all_pairs(tasks: List[Task]) -> List[Tuple[int, int]]:
    """The same relation by comparing every task with every task (used on
    tiny graphs to check the per-tensor grouping)."""
    pairs = set()
    for p in tasks:
        for c in tasks:
            if p.id != c.id and any(_overlap(w, r) for w in p.writes
                                    for r in c.reads):
                pairs.add((p.id, c.id))
    return sorted(pairs)


def fuse(raw: List[Tuple[int, int]]) -> Dict[int, Tuple[set, set]]:
    """Def 4.1 (equal OutTasks -> union InTasks) then Def 4.2 (equal InTasks
    -> union OutTasks), repeated until a full round changes nothing.
    Returns {event id: (InTasks, OutTasks)}; the survivor of a merge is the
    member with the smallest id."""
    ev = {i: ({p}, {c}) for i, (p, c) in enumerate(raw)}
    changed = True
    while changed:
        changed = False
        for which in (1, 0):          # 1: group by OutTasks (Def 4.1)
            groups = collections.defaultdict(list)
            for i in sorted(ev):
                groups[frozenset(ev[i][which])].append(i)
            for ids in groups.values():
                if len(ids) < 2:
                    continue
                keep = ids[0]
                other = 1 - which
                merged = set()
                for i in ids:
                    merged |= ev[i][other]
                ins, outs = ev[keep]
                if which == 1:
                    ev[keep] = (merged, outs)
                else:
                    ev[keep] = (ins, merged)
                for i in ids[1:]:
                    del ev[i]
                changed = True
    return ev


@dataclasses.dataclass
class Graph:
    ops: List[Op]
    tasks: List[Task]             # indexed by pre-linearisation id
    n_chunks: int
    kinds: List[str]              # per pre-linearisation task id
    # after linearisation
    order: List[int]              # linear position -> task id
    task_pos: Dict[int, int]
    event_order: List[int]        # linear event id -> pre-lin event id
    dep: List[int]                # per linear task: linear event id
    trig: List[int]
    launch: List[int]
    worker: List[int]
    ev_count: List[int]
    ev_first: List[int]
    ev_last: List[int]
    n_empty: int
    raw: List[Tuple[int, int]]
    fused: Dict[int, Tuple[set, set]]


def build(shape, batch: int, max_ctx: int, tiles: Tiles) -> Graph:
    """Decompose a decoder step and run every pass on it."""
    ops, tasks, C = decompose(shape, batch, max_ctx, tiles)
    jit = () if attn_is_aot(batch, max_ctx, C) else ("attn",)
    return build_from_tasks(ops, tasks, tiles.num_workers, C, jit)


def build_from_tasks(ops: List[Op], tasks: List[Task], num_workers: int,
                     n_chunks: int = 0, jit_kinds=("attn",)) -> Graph:
    """Dependencies, fusion, normalisation, linearisation and AOT assignment
    for an already decomposed task list (tasks[i].id == i)."""
    raw = raw_events(tasks)
    fused = fuse(raw)
    kinds = [t.kind for t in tasks]
    g = normalize_and_linearize(kinds, fused, num_workers, jit_kinds)
    g.ops, g.n_chunks, g.raw, g.fused = ops, n_chunks, raw, fused
    g.tasks = list(tasks) + [
        Task(id=i, op=-1, kind="empty", layer=-1, tile=0)
        for i in range(len(tasks), len(g.kinds))]
    return g


def normalize_and_linearize(kinds: List[str],
                            fused: Dict[int, Tuple[set, set]],
                            num_workers: int,
                            jit_kinds=("attn",)) -> "Graph":
    """Normalisation, root/end events, BFS linearisation and AOT assignment
    on fused events {id: (InTasks, OutTasks)} over tasks 0..len(kinds)-1."""
    ev = {i: (set(a), set(b)) for i, (a, b) in fused.items()}
    next_ev = (max(ev) + 1) if ev else 0
    kinds = list(kinds)
    n_real = len(kinds)

    def new_empty():
        kinds.append("empty")
        return len(kinds) - 1

    trig_sets = collections.defaultdict(set)    # task -> events it triggers
    dep_sets = collections.defaultdict(set)     # task -> events it waits on
    for i, (ins, outs) in ev.items():
        for t in ins:
            trig_sets[t].add(i)
        for t in outs:
            dep_sets[t].add(i)

    # fan-out: a task triggering k > 1 events triggers one new event e';
    # k empty tasks wait on e' and each triggers one of the old events
    for t in range(n_real):
        trig = sorted(trig_sets[t])
        if len(trig) > 1:
            e1 = next_ev
            next_ev += 1
            ev[e1] = ({t}, set())
            trig_sets[t] = {e1}
            for ei in trig:
                Ti = new_empty()
                ev[ei][0].discard(t)
                ev[ei][0].add(Ti)
                ev[e1][1].add(Ti)
                trig_sets[Ti] = {ei}
                dep_sets[Ti] = {e1}
    # fan-in: a task waiting on k > 1 events waits on one new event e'';
    # k empty tasks each wait on one of the old events and trigger e''
    for t in range(len(kinds)):
        deps = sorted(dep_sets[t])
        if len(deps) > 1:
            e2 = next_ev
            next_ev += 1
            ev[e2] = (set(), {t})
            dep_sets[t] = {e2}
            for ei in deps:
                Ti = new_empty()
                ev[ei][1].discard(t)
                ev[ei][1].add(Ti)
                ev[e2][0].add(Ti)
                dep_sets[Ti] = {ei}
                trig_sets[Ti] = {e2}

    nT = len(kinds)
    dep_map = {}
    trig_map = {}
    for i, (ins, outs) in ev.items():
        for t in outs:
            assert t not in dep_map
            dep_map[t] = i
        for t in ins:
            assert t not in trig_map
            trig_map[t] = i
    root = next_ev
    end = next_ev + 1
    ev[root] = (set(), {t for t in range(nT) if t not in dep_map})
    ev[end] = ({t for t in range(nT) if t not in trig_map}, set())
    for t in ev[root][1]:
        dep_map[t] = root
    for t in ev[end][0]:
        trig_map[t] = end

    # Kahn-style BFS linearisation from the root
    remaining = {i: len(ins) for i, (ins, _) in ev.items()}
    queue = collections.deque([root])
    event_order, order = [], []
    ev_first, ev_last = {}, {}
    while queue:
        e = queue.popleft()
        event_order.append(e)
        outs = sorted(ev[e][1])
        ev_first[e] = len(order)
        order.extend(outs)
        ev_last[e] = len(order) - 1
        for t in outs:
            te = trig_map[t]
            remaining[te] -= 1
            if remaining[te] == 0:
                queue.append(te)
    assert len(order) == nT and len(event_order) == len(ev), \
        "linearisation did not reach every task and event"
    ev_pos = {e: i for i, e in enumerate(event_order)}
    task_pos = {t: i for i, t in enumerate(order)}

    launch, worker = [], []
    k = 0
    for t in order:
        kind = kinds[t]
        if kind == "empty":
            launch.append(INLINE)
            worker.append(-1)
        elif kind in jit_kinds:
            launch.append(JIT)
            worker.append(-1)
        else:
            launch.append(AOT)
            worker.append(k % num_workers)
            k += 1
    return Graph(
        ops=[], tasks=[], n_chunks=0, kinds=kinds, order=order,
        task_pos=task_pos, event_order=event_order,
        dep=[ev_pos[dep_map[t]] for t in order],
        trig=[ev_pos[trig_map[t]] for t in order],
        launch=launch, worker=worker,
        ev_count=[len(ev[e][0]) for e in event_order],
        ev_first=[ev_first[e] for e in event_order],
        ev_last=[ev_last[e] for e in event_order],
        n_empty=nT - n_real, raw=[], fused={})
