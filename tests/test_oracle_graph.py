"""Pins for the oracle tGraph builder (CPU only): hand-worked fixtures and
the properties the pages fix (MPK: A Compiler and Runtime for
Mega-Kernelizing Tensor Programs, §4 "6 minimum checks", Defs 4.1/4.2)."""
import collections
import os
import random

import pytest

from oracle import tgraph
from task_graph_runtime_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_region(s):
    name, r0, r1, c0, c1 = s.split(":")
    return (name, int(r0), int(r1), int(c0), int(c1))


def load_fixture(fname):
    tasks, fused, exp = [], {}, {}
    ntasks = None
    for line in open(os.path.join(GOLDEN, fname)):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "task":
            tid, kind = int(f[1]), f[2]
            reads = [] if f[4] == "-" else [_parse_region(r)
                                              for r in f[4].split(",")]
            writes = [_parse_region(r) for r in f[6].split(",")]
            tasks.append(tgraph.Task(id=tid, op=0, kind=kind, layer=0, tile=0,
                                     reads=reads, writes=writes))
        elif f[0] == "ntasks":
            ntasks = int(f[1])
        elif f[0] == "raw":
            exp["raw"] = [tuple(int(x) for x in p.split(",")) for p in f[1:]]
        elif f[0] == "fused":
            fused[int(f[1])] = ({int(x) for x in f[3].split(",")},
                                {int(x) for x in f[5].split(",")})
        else:
            exp[f[0]] = [int(x) for x in f[1:]]
    return tasks, ntasks, fused, exp


def test_golden_fusion_and_fanout():
    tasks, _, fused, exp = load_fixture("fusion_fanout.txt")
    assert tgraph.raw_events(tasks) == exp["raw"]
    assert tgraph.raw_events_all_pairs(tasks) == exp["raw"]
    got = tgraph.fuse(exp["raw"])
    assert {k: (set(a), set(b)) for k, (a, b) in got.items()} == fused
    g = tgraph.build_from_tasks([], tasks, num_workers=2)
    for key in ("order", "dep", "trig", "count", "first", "last"):
        val = {"order": g.order, "dep": g.dep, "trig": g.trig,
               "count": g.ev_count, "first": g.ev_first,
               "last": g.ev_last}[key]
        assert val == exp[key], key
    assert g.n_empty == 4


def test_golden_fanin():
    _, ntasks, fused, exp = load_fixture("fanin.txt")
    g = tgraph.normalize_and_linearize(["x"] * ntasks, fused, 1)
    assert g.order == exp["order"]
    assert g.dep == exp["dep"] and g.trig == exp["trig"]
    assert g.ev_count == exp["count"]
    assert g.ev_first == exp["first"] and g.ev_last == exp["last"]
    assert g.n_empty == 2


# ------------------------------------------------------------ properties
def _reach(n, edges):
    """Transitive closure as bitsets: reach[u] = set of v reachable from u."""
    succ = collections.defaultdict(set)
    for u, v in edges:
        succ[u].add(v)
    order = _topo(n, succ)
    reach = [0] * n
    for u in reversed(order):
        r = 0
        for v in succ[u]:
            r |= (1 << v) | reach[v]
        reach[u] = r
    return reach


def _topo(n, succ):
    indeg = [0] * n
    for u in succ:
        for v in succ[u]:
            indeg[v] += 1
    q = collections.deque(i for i in range(n) if indeg[i] == 0)
    out = []
    while q:
        u = q.popleft()
        out.append(u)
        for v in succ[u]:
            indeg[v] -= 1
            if indeg[v] == 0:
                q.append(v)
    assert len(out) == n, "cycle"
    return out


def _graph_edges(g):
    """Task-level edges of the final graph, in pre-linearisation ids:
    every producer of an event precedes every consumer of it."""
    prods = collections.defaultdict(list)
    cons = collections.defaultdict(list)
    for pos, t in enumerate(g.order):
        prods[g.trig[pos]].append(t)
        cons[g.dep[pos]].append(t)
    return [(p, c) for e in prods for p in prods[e] for c in cons[e]]


SMALL_CASES = [
    ("tiny", synth.WORKLOADS["tiny"].shape, 1, 144, tgraph.Tiles(4)),
    ("tiny_w7", synth.WORKLOADS["tiny"].shape, 1, 144, tgraph.Tiles(7)),
    ("tiny_b3", synth.WORKLOADS["tiny"].shape, 3, 144,
     tgraph.Tiles(5, attn_chunks=3)),
    ("tiny_r24", synth.WORKLOADS["tiny"].shape, 2, 144,
     tgraph.Tiles(6, gemv_rows_per_task=24, attn_chunks=2)),
    ("tiny_c1_jit", synth.WORKLOADS["tiny"].shape, 1, 144,
     tgraph.Tiles(4, attn_chunks=1)),
    ("tiny_coarse", synth.WORKLOADS["tiny"].shape, 1, 144,
     tgraph.Tiles(4, coarse_events=1)),
    ("tiny_b8_mma", synth.WORKLOADS["tiny"].shape, 8, 144,
     tgraph.Tiles(5, mma_rows_per_task=16)),
    ("chain", synth.ModelShape(0, 64, 1, 1, 32, 0, 96, chain_ffn=160), 2, 0,
     tgraph.Tiles(3)),
]


@pytest.fixture(scope="module", params=SMALL_CASES, ids=lambda c: c[0])
def built(request):
    _, shape, B, ctx, tiles = request.param
    return tgraph.build(shape, B, ctx, tiles)


def test_overlap_grouping_equals_all_pairs(built):
    real = [t for t in built.tasks if t.kind != "empty"]
    assert tgraph.raw_events(real) == tgraph.raw_events_all_pairs(real)


def test_fusion_leaves_no_equal_sets(built):
    outs = [frozenset(o) for _, o in built.fused.values()]
    ins = [frozenset(i) for i, _ in built.fused.values()]
    assert len(set(outs)) == len(outs), "Def 4.1 not applied to a fixpoint"
    assert len(set(ins)) == len(ins), "Def 4.2 not applied to a fixpoint"


def test_dependencies_preserved_exactly(built):
    """Every raw producer->consumer edge is implied by the final graph, and
    the final graph implies no dependency between real tasks that the raw
    graph did not have."""
    nT = len(built.tasks)
    n_real = nT - built.n_empty
    raw_reach = _reach(nT, built.raw)
    fin_reach = _reach(nT, _graph_edges(built))
    mask = (1 << n_real) - 1
    for u in range(n_real):
        assert fin_reach[u] & mask == raw_reach[u] & mask, u


def test_normalised_and_contiguous(built):
    nE = len(built.ev_count)
    consumers = collections.defaultdict(list)
    producers = collections.defaultdict(list)
    for pos in range(len(built.order)):
        consumers[built.dep[pos]].append(pos)
        producers[built.trig[pos]].append(pos)
    for e in range(nE):
        cs = consumers[e]
        assert cs == list(range(built.ev_first[e], built.ev_last[e] + 1))
        assert built.ev_count[e] == len(producers[e])
        # topological: every producer precedes every consumer
        if cs and producers[e]:
            assert max(producers[e]) < min(cs)
    assert built.ev_count[0] == 0                    # root
    assert built.ev_last[-1] == built.ev_first[-1] - 1   # end: no consumers
    assert sorted(built.order) == list(range(len(built.order)))


def test_launch_classes_and_aot_round_robin(built):
    """Empty tasks inline; attention chunks JIT unless they are equal and
    small (batch 1, <= 128 tokens); every other task AOT, dealt round-robin
    in linear order (MPK summary, "Design space": hybrid JIT/AOT)."""
    k = 0
    W = max(w for w in built.worker) + 1
    kinds = {built.tasks[t].kind for t in built.order}
    attn_jit = None
    for pos, t in enumerate(built.order):
        kind = built.tasks[t].kind
        if kind == "empty":
            assert built.launch[pos] == tgraph.INLINE
            continue
        if kind == "attn":
            jit = built.launch[pos] == tgraph.JIT
            assert attn_jit in (None, jit)     # one class for the operator
            attn_jit = jit
            if jit:
                assert built.worker[pos] == -1
                continue
        assert built.launch[pos] == tgraph.AOT
        assert built.worker[pos] == k % W
        k += 1
    if "attn" in kinds:
        n_attn = sum(1 for t in built.tasks if t.kind == "attn")
        B = 1 + max(t.b for t in built.tasks if t.kind == "attn")
        assert attn_jit == (B > 1 or built.n_chunks == 1)


def test_row_tiles_cover_rows():
    """Default tiles: contiguous, multiples of the unit, within the cap, a
    multiple of W of them unless every tile is one unit, sizes within one
    unit of each other."""
    for unit in (1, 8):
        for n in (8, 64, 688, 1000, 6144, 12288, 151936):
            for W in (1, 7, 148):
                for cap in (32, 64, 128, 1024, 2048):
                    tl = tgraph.row_tiles(n, 0, W, cap, unit)
                    assert tl[0][0] == 0 and tl[-1][1] == n
                    assert all(a[1] == b[0] for a, b in zip(tl, tl[1:]))
                    assert all(r0 % unit == 0 and r1 > r0 for r0, r1 in tl)
                    assert all(r1 - r0 <= cap for r0, r1 in tl)
                    U = -(-n // unit)
                    assert len(tl) % W == 0 or len(tl) == U
                    sizes = [r1 - r0 for r0, r1 in tl[:-1]]
                    if sizes:
                        assert max(sizes) - min(sizes) <= unit


def test_tile_caps_by_batch():
    assert tgraph.tile_row_cap(1, False, 4096) == 1280     # 4 rows/page, 2 warps/row
    assert tgraph.tile_row_cap(1, True, 4096) == 640
    assert tgraph.tile_row_cap(1, False, 12288) == 320     # 1 row/page, 8 parts
    assert tgraph.tile_row_cap(1, False, 8192) == 640      # 2 rows/page, 4 parts
    assert tgraph.tile_row_cap(1, False, 6144) == 640      # 2 rows/page, 4 parts
    assert tgraph.tile_row_cap(1, False, 688) == 2560      # 23 rows/page
    assert tgraph.tile_row_cap(1, False, 2048) == 2560     # 8 rows/page
    assert tgraph.tile_row_cap(1, False, 256) == 2560
    assert tgraph.tile_row_cap(4, False, 4096) == 64
    assert tgraph.tile_row_cap(16, True, 12288) == 64


def test_coarse_events_are_operator_level():
    """Figure 4c: with operator-level events every task of an operator
    waits for every task of each operator it reads, so one event separates
    consecutive operators."""
    shape = synth.WORKLOADS["tiny"].shape
    fine = tgraph.build(shape, 1, 144, tgraph.Tiles(4))
    coarse = tgraph.build(shape, 1, 144, tgraph.Tiles(4, coarse_events=1))
    assert (len(coarse.order) - coarse.n_empty ==
            len(fine.order) - fine.n_empty)
    # every attention chunk of layer 0 waits on the event the whole qkv
    # operator triggers (fine: only on the tiles holding its head's columns)
    attn = [p for p, t in enumerate(coarse.order)
            if coarse.tasks[t].kind == "attn" and coarse.tasks[t].layer == 0]
    deps = {coarse.dep[p] for p in attn}
    assert len(deps) == 1
    qkv0 = [t for t in coarse.tasks if t.kind == "qkv" and t.layer == 0]
    e = deps.pop()
    assert coarse.ev_count[e] >= len(qkv0)
    fine_attn = [p for p, t in enumerate(fine.order)
                 if fine.tasks[t].kind == "attn" and fine.tasks[t].layer == 0]
    assert len({fine.dep[p] for p in fine_attn}) > 1


def test_random_chains_properties():
    """Random small operator chains with random tilings and region shapes."""
    rnd = random.Random(5)
    for trial in range(25):
        tasks = []
        n_cols = rnd.choice([4, 6, 8])
        prev = None
        for op in range(rnd.randint(2, 5)):
            nt = rnd.randint(1, 4)
            cuts = sorted(rnd.sample(range(1, n_cols), min(nt - 1, n_cols - 1)))
            bounds = [0] + cuts + [n_cols]
            for i in range(len(bounds) - 1):
                reads = []
                if prev is not None:
                    if rnd.random() < 0.5:
                        reads = [(prev, 0, 1, 0, n_cols)]
                    else:
                        a = rnd.randrange(n_cols)
                        reads = [(prev, 0, 1, a, rnd.randint(a + 1, n_cols))]
                tasks.append(tgraph.Task(id=len(tasks), op=op, kind="x",
                                         layer=0, tile=i, reads=reads,
                                         writes=[(f"T{op}", 0, 1, bounds[i],
                                                  bounds[i + 1])]))
            prev = f"T{op}"
        g = tgraph.build_from_tasks([], tasks, num_workers=3)
        assert tgraph.raw_events(tasks) == tgraph.raw_events_all_pairs(tasks)
        nT = len(g.kinds)
        raw_reach = _reach(nT, g.raw)
        fin_reach = _reach(nT, _graph_edges(g))
        mask = (1 << len(tasks)) - 1
        for u in range(len(tasks)):
            assert fin_reach[u] & mask == raw_reach[u] & mask
        for e in range(len(g.ev_count)):
            cs = [p for p in range(len(g.order)) if g.dep[p] == e]
            assert cs == list(range(g.ev_first[e], g.ev_last[e] + 1))


def test_overlap_is_strict_on_both_axes():
    """Half-open rectangles that only touch share no element: no event.  A
    single shared element is an overlap: one event (MegaKernel HN comments,
    point 2: a dependency iff A produces any element B consumes)."""
    def mk(i, reads, writes):
        return tgraph.Task(id=i, op=0, kind="x", layer=0, tile=0,
                           reads=reads, writes=writes)
    touching = [mk(0, [], [("X", 0, 2, 0, 2)]),
                mk(1, [("X", 2, 4, 0, 2)], [("Y", 0, 1, 0, 1)]),
                mk(2, [("X", 0, 2, 2, 4)], [("Y", 0, 1, 1, 2)]),
                mk(3, [("Z", 0, 2, 0, 2)], [("Y", 0, 1, 2, 3)])]
    assert tgraph.raw_events(touching) == []
    mirrored = [mk(0, [], [("X", 2, 4, 2, 4)]),
                mk(1, [("X", 0, 2, 2, 4)], [("Y", 0, 1, 0, 1)]),
                mk(2, [("X", 2, 4, 0, 2)], [("Y", 0, 1, 1, 2)])]
    assert tgraph.raw_events(mirrored) == []
    assert tgraph.raw_events_all_pairs(mirrored) == []
    one_cell = [mk(0, [], [("X", 0, 2, 0, 2)]),
                mk(1, [("X", 1, 4, 1, 3)], [("Y", 0, 1, 0, 1)]),
                mk(2, [("X", 1, 2, 1, 2)], [("Y", 0, 1, 1, 2)]),
                mk(3, [("X", 2, 3, 1, 2)], [("Y", 0, 1, 2, 3)])]
    assert tgraph.raw_events(one_cell) == [(0, 1), (0, 2)]
    assert tgraph.raw_events_all_pairs(one_cell) == [(0, 1), (0, 2)]
